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
//      lower-triangular inverse T in 16x16 blocks, W and Ut, the masked,
//      decayed P = M o Q K^T and dec o K; they go to the workspace already in
//      the scan's operand-tile layout (128.25 KB per chunk and head).
//  (2) gdn_chunk_scan_kernel -- one CTA per (sequence, v-head): the only
//      sequential part.  The state stays on chip across the sequence's
//      chunks; per chunk it forms U, the outputs and the next state.
// Sequence i's chunks start at cu_seqlens[i]; chunk c of sequence i uses
// workspace slot (cu_seqlens[i] + 64c)/64 + i, unique and below
// ceil(row_capacity/64) + nseq.
#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace {

constexpr int kC = 64;         // chunk length
constexpr int kD = 128;        // d_k = d_v supported by this kernel pair
constexpr int kThreads = 256;       // per-chunk kernel
constexpr int kScanThreads = 512;   // scan: 4 warps per tensor-memory lane quadrant

__device__ __forceinline__ int chunk_slot(int seq_start, int c, int seq) { return (seq_start + kC * c) / kC + seq; }

struct PrefArgs {
    const int32_t *cu;
    int32_t nseq, h_qk, h_v, grp, row_capacity, num_slots;
    const uint16_t *q, *k, *v;
    const float *g, *beta;
    float *pool;
    int64_t slot_stride;
    const int32_t *src_slot, *dst_slot;
    uint16_t *o;
    float *ws;             // per (chunk slot, v-head) blobs, see namespace blob
    const int32_t *order;      // sequences by decreasing length (written by gdn_prefill_tables_kernel)
    const int32_t *chunk_seq;  // per chunk slot: its sequence, or -1 (same kernel)
    float q_scale;
    uint32_t *status;
    // q, k (rows x h_qk x 128) and v (rows x h_v x 128) as 3-D bf16 tensors
    // for the copy engine: boxes of 64 columns x 1 head x 64 rows, 128-byte
    // swizzle, zero fill past row_capacity
    CUtensorMap tm_q, tm_k, tm_v;
};

// Workspace per (chunk slot, v-head): everything the scan needs for one chunk,
// written by the per-chunk kernel in the scan's own shared-memory layout so
// that the scan fetches it with bulk copies and starts its products at once.
// Operand tiles are 128-byte-swizzled K-major bf16 tiles (tc.cuh); "parts"
// are the two-term bf16 split x = x1 + x2, x1 = bf16(x), x2 = bf16(x - x1).
namespace blob {
// [W1; Q]: W's high part (rows 0..63) stacked on Q (exact bf16, rows 64..127),
// one 128-row tile (atoms 16 KB apart) so that one N = 128 product gives
// S W1^T and S Q^T together; W's low part W2 is a 64-row tile.
constexpr uint32_t kW1Q = 0;                 // 128 rows (t, then t) x 128 (d_k)
constexpr uint32_t kW2 = 32768;              // 64 rows (t) x 128 (d_k)
constexpr uint32_t kP1 = 49152, kP2 = 57344; // P = M o Q K^T parts:         64 rows (t) x  64 (i)
constexpr uint32_t kK1 = 65536, kK2 = 81920; // dec o K parts, MN-major B:  64 rows (i) x 128 (d_k)
constexpr uint32_t kTiles = 98304;           // bytes of operand tiles (one contiguous block)
constexpr uint32_t kUt = 98304;              // Ut = T diag(beta) V, fp32 [t][d_v] (pieces permuted, ut_index)
constexpr uint32_t kEG = 131072;             // e^{G_t}, fp32 x 64
constexpr uint32_t kBytes = 131328;
}  // namespace blob
constexpr size_t kWsFloats = blob::kBytes / 4;

// G[t] = g[0] + ... + g[t] over the chunk (g = 0 past its n tokens), by warp 0
// with a shuffle scan.
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

__device__ __forceinline__ unsigned char *ws_blob(const PrefArgs &a, int slot, int h) {
    return reinterpret_cast<unsigned char *>(a.ws) + (size_t(slot) * a.h_v + h) * blob::kBytes;
}

// x0 and x1 rounded to nearest-even bf16, packed with x0 in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float x0, float x1) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(x1), "f"(x0));
    return d;
}

// e^x for the gates inside a chunk (x <= 0): 2^(x log2 e).
__device__ __forceinline__ float gate_exp(float x) { return exp2f(x * 1.4426950408889634f); }

// Two-term bf16 split of 8 consecutive values, packed as two 16-byte chunks.
__device__ __forceinline__ void split8(const float *x, uint4 &hi, uint4 &lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        h[p] = pack_bf16x2(x[2 * p], x[2 * p + 1]);
        l[p] = pack_bf16x2(x[2 * p] - __uint_as_float(h[p] << 16), x[2 * p + 1] - __uint_as_float(h[p] & 0xffff0000u));
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// ---------------------------------------------------------------------------
// (1) per-chunk WY/UT quantities on the tensor cores (tcgen05, kind::f16)
// ---------------------------------------------------------------------------
// Shared-memory map (bytes from a 1024-aligned base), bf16 128-byte-swizzled tiles:
//   A1   [K; Q]   128 rows (tokens, then q rows) x 128 (d_k), K-major   32 KB
//   VN   V        64 rows (tokens) x 128 (d_v) in two 64-column atoms 16 KB
//                 apart, right after A1: with the K rows of A1 this is
//                 [K | V] as an MN-major B operand (N = 256, 64-element
//                 blocks 16 KB apart), so no transposed copy is needed
//   AB   [T diag(beta e^G); T diag(beta)], hi and lo parts,
//                 128 rows (t, twice) x 64 (i), K-major                2 x 16 KB
//   (the fp32 matrix A -> T, [64][68], lives in the AB area before those
//    tiles are written)
//   misc G, beta, e^G, mbarrier, tensor-memory base, flag, dec
// Outputs: the Q tile (rows 64..127 of both A1 atoms as the copy engine left
// them) leaves by bulk copies once the first product is done, and the P and
// dec o K parts go from registers straight to the workspace; the W and Ut
// parts are staged (the W parts in the K rows of A1 and the V rows of VN,
// both consumed by the second product, Ut where AB was) and leave by bulk
// copies at the very end: written from registers, their rows would scatter.
// Tensor memory (256 columns): first D1 = [K;Q] K^T at columns 0..63 (rows
// 0..63: K K^T, rows 64..127: Q K^T), then D2 = AB [K | V] at 0..255:
// rows 0..63 x columns 0..127 hold W, rows 64..127 x columns 128..255 hold Ut
// (the two cross blocks are not used).
namespace wy {
constexpr uint32_t kA1 = 0, kVN = 32768, kT = 65536, kMisc = 98304;
constexpr uint32_t kAbHi = kT, kAbLo = kT + 16384;
// Staging (8 KB pieces): the two 64-column atoms of W1 in the K rows of the
// A1 atoms and those of W2 in the V rows of the VN atoms; Ut in AB.
__device__ __forceinline__ uint32_t st_w1(int atom) { return kA1 + 16384u * uint32_t(atom); }
__device__ __forceinline__ uint32_t st_w2(int atom) { return kVN + 16384u * uint32_t(atom); }
constexpr uint32_t kStUt = kT;  // 32 KB
constexpr int kAs = 68;         // row stride (floats) of the fp32 matrix A -> T: 16-byte rows, no bank conflicts
constexpr size_t kSmem = kMisc + 2048 + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 256;
}  // namespace wy

// Ut in the workspace: fp32 rows t of 128 values whose 16-byte pieces are
// permuted within each 128-byte segment by (piece ^ (t & 7)), so that the
// per-chunk kernel stages it without bank conflicts while a warp of the scan
// still reads 32 consecutive values of one row from one segment.
__host__ __device__ constexpr int ut_index(int t, int j) { return t * kD + ((((j >> 2) ^ (t & 7))) << 2) + (j & 3); }

__global__ void __launch_bounds__(kThreads) gdn_chunk_wy_kernel(const __grid_constant__ PrefArgs a) {
    // One CTA per chunk slot and v-head; slots that hold no chunk exit.
    const int seq = a.chunk_seq[blockIdx.x];
    if (seq < 0) return;
    const int h = blockIdx.y;
    const int s0 = a.cu[seq];
    const int s1 = a.cu[seq + 1];
    const int len = s1 - s0;
    if (s0 < 0 || len < 0 || s1 > a.row_capacity) return;  // reported by the scan kernel
    const int c = int(blockIdx.x) - seq - s0 / kC;         // inverse of chunk_slot
    if (c < 0 || c * kC >= len) return;
    const int t0 = s0 + c * kC;
    const int n = min(kC, len - c * kC);
    const int hq = h / a.grp;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned char *out = ws_blob(a, chunk_slot(s0, c, seq), h);

    extern __shared__ unsigned char smraw[];
    const uint32_t raw_u = gdn::smem_u32(smraw);
    unsigned char *sm = smraw + (((raw_u + 1023u) & ~1023u) - raw_u);
    const uint32_t sb = gdn::smem_u32(sm);
    float *Af = reinterpret_cast<float *>(sm + wy::kT);
    float *Gs = reinterpret_cast<float *>(sm + wy::kMisc);
    float *Bs = Gs + kC;
    float *eG = Bs + kC;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + wy::kMisc + 768);
    uint32_t *tbase = reinterpret_cast<uint32_t *>(sm + wy::kMisc + 776);
    int *flag = reinterpret_cast<int *>(sm + wy::kMisc + 780);
    float *dec = reinterpret_cast<float *>(sm + wy::kMisc + 1024);

    uint64_t *bar_ld = reinterpret_cast<uint64_t *>(sm + wy::kMisc + 784);
    int *staged_flag = reinterpret_cast<int *>(sm + wy::kMisc + 792);

    // Stage K, Q (rows of A1) and V (rows of VN) by six tensor copies of
    // 64 rows x 64 columns each, 128-byte swizzled by the copy engine (the
    // layout of the operand tiles); the gates by the threads meanwhile.
    if (tid == 0) {
        gdn::mbar_init(bar, 1);
        gdn::mbar_init(bar_ld, 1);
        gdn::mbar_arrive_expect_tx(bar_ld, 6u * 8192u);
#pragma unroll
        for (int at = 0; at < 2; ++at) {
            gdn::tma_load_3d(sm + wy::kA1 + at * 16384, &a.tm_k, 64 * at, hq, t0, bar_ld);
            gdn::tma_load_3d(sm + wy::kA1 + at * 16384 + 8192, &a.tm_q, 64 * at, hq, t0, bar_ld);
            gdn::tma_load_3d(sm + wy::kVN + at * 16384, &a.tm_v, 64 * at, h, t0, bar_ld);
        }
    }
    __syncwarp();
    if (warp == 0) tc::tmem_alloc(tbase, wy::kTmemCols);
    if (tid < kC) {
        Bs[tid] = tid < n ? a.beta[size_t(t0 + tid) * a.h_v + h] : 0.f;
        Gs[tid] = tid < n ? a.g[size_t(t0 + tid) * a.h_v + h] : 0.f;
    }
    if (tid == 0) *staged_flag = gdn::mbar_wait_bounded(bar_ld, 0) ? 1 : 0;
    __syncthreads();
    const bool staged = *staged_flag != 0;
    if (staged && n < kC) {
        // Rows n..63 (the next sequence's rows or padding) become zero: K,
        // Q and V rows, 128 bytes per row and atom.
        for (int e = tid; e < (kC - n) * 48; e += kThreads) {
            const int piece = e & 7, rest = e >> 3;
            const int which = rest % 6, row = n + rest / 6;
            const uint32_t off = which < 4 ? wy::kA1 + (which >> 1) * 16384 + (which & 1) * 8192
                                           : wy::kVN + (which - 4) * 16384;
            *reinterpret_cast<uint4 *>(sm + off + row * 128 + piece * 16) = make_uint4(0, 0, 0, 0);
        }
    }
    gdn::fence_proxy_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tbase;

    // D1 = A1 K^T: rows 0..63 are K K^T, rows 64..127 are Q K^T.
    if (tid == 0 && staged) {
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
        // While the product runs: G = cumsum(g) (in place: each lane owns two
        // entries), e^G and dec_i = e^{G_last - G_i} (0 past the n tokens).
        chunk_cumsum(Gs, n, Gs);
        __syncwarp();
        const float gl = Gs[n - 1];
#pragma unroll
        for (int e = lane; e < kC; e += 32) {
            const float ge = Gs[e];
            const float x = expf(ge);
            eG[e] = x;
            dec[e] = e < n ? expf(gl - ge) : 0.f;
            reinterpret_cast<float *>(out + blob::kEG)[e] = x;
        }
        if (lane == 0) *flag = staged && gdn::mbar_wait_bounded(bar, 0) ? 1 : 0;
    }
    __syncthreads();
    bool ok = *flag != 0;
    if (ok) {
        (void)gdn::mbar_try_wait(bar, 0);
        tc::fence_after();
        if (tid == 0) {
            // The Q tile as it stands; the copy is done long before the
            // second product is issued.
            gdn::bulk_s2g(out + blob::kW1Q + 8192, sm + wy::kA1 + 8192, 8192u);
            gdn::bulk_s2g(out + blob::kW1Q + 16384 + 8192, sm + wy::kA1 + 16384 + 8192, 8192u);
            gdn::bulk_commit();
        }
        // Rows 0..63: A[t][i] = beta_t e^{G_t-G_i} (k_t.k_i), i < t (0 elsewhere).
        // Rows 64..127: P[t][i] = e^{G_t-G_i} (q_t.k_i), i <= t, split into its
        // two parts in the staging area (rows 0..63 of the A1 atoms: the K rows,
        // consumed by the product above).
        // Masked entries take e^{-inf} = 0 (K and Q rows past n are zero, so
        // every product is finite): no divergent branch per element.
        const int q4 = warp & 3, hc = warp >> 2;
        const int t = 32 * (q4 & 1) + lane;
        const float gt = Gs[t], bt = Bs[t];
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            float v16[16];
            const int col0 = 32 * hc + 16 * part;
            tc::ld16(tm + (uint32_t(32 * q4) << 16) + uint32_t(col0), v16);
            if (q4 < 2) {
#pragma unroll
                for (int x = 0; x < 16; x += 4) {
                    float av[4];
#pragma unroll
                    for (int y = 0; y < 4; ++y) {
                        const int i = col0 + x + y;
                        av[y] = bt * gate_exp(i < t && t < n ? gt - Gs[i] : -INFINITY) * v16[x + y];
                    }
                    *reinterpret_cast<float4 *>(Af + t * wy::kAs + col0 + x) = make_float4(av[0], av[1], av[2], av[3]);
                }
            } else {
                float pe[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const int i = col0 + x;
                    pe[x] = gate_exp(i <= t && t < n ? gt - Gs[i] : -INFINITY) * v16[x];
                }
#pragma unroll
                for (int x = 0; x < 16; x += 8) {
                    uint4 hi, lo;
                    split8(pe + x, hi, lo);
                    const uint32_t off = tc::swz_off(64, t, col0 + x);
                    *reinterpret_cast<uint4 *>(out + blob::kP1 + off) = hi;
                    *reinterpret_cast<uint4 *>(out + blob::kP2 + off) = lo;
                }
            }
        }
        gdn::fence_proxy_async_smem();
    }
    __syncthreads();
    if (ok) {
        // T = (I + A)^{-1} by forward substitution, column by column, four
        // pivot rows at a time: T[t][j] = delta_tj - sum_{i<t} A[t][i] T[i][j].
        // Four threads own a column j (rows 4m + q, m = 0..15) and keep the
        // running sums p of their rows.  For pivot rows 4 tau .. 4 tau + 3 the
        // owners' right-hand sides b = delta - p go to all four threads, which
        // solve the unit lower-triangular 4 x 4 diagonal block of (I + A) in
        // closed form (D = its inverse) and add A[r][4 tau .. 4 tau + 3] v to
        // the sums of their later rows r.  Pivots above a warp's first column
        // give zeros and are skipped; column blocks are assigned so that the
        // two warps sharing a scheduler (w, w + 4) have the same number of steps.
        {
            const int cb = warp < 4 ? warp : 11 - warp;
            const int j = 8 * cb + (lane >> 2), q = lane & 3;
            const int base = lane & ~3;
            float p[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) p[m] = 0.f;
#pragma unroll
            for (int tau = 0; tau < 16; ++tau) {
                if (tau >= 2 * cb) {
                    const float4 a1 = *reinterpret_cast<const float4 *>(Af + (4 * tau + 1) * wy::kAs + 4 * tau);
                    const float4 a2 = *reinterpret_cast<const float4 *>(Af + (4 * tau + 2) * wy::kAs + 4 * tau);
                    const float4 a3 = *reinterpret_cast<const float4 *>(Af + (4 * tau + 3) * wy::kAs + 4 * tau);
                    const float d10 = -a1.x, d21 = -a2.y, d32 = -a3.z;
                    const float d20 = -fmaf(a2.y, d10, a2.x);
                    const float d31 = -fmaf(a3.z, d21, a3.y);
                    const float d30 = -fmaf(a3.z, d20, fmaf(a3.y, d10, a3.x));
                    const float bq = (4 * tau + q == j ? 1.f : 0.f) - p[tau];
                    const float b0 = __shfl_sync(0xffffffffu, bq, base);
                    const float b1 = __shfl_sync(0xffffffffu, bq, base | 1);
                    const float b2 = __shfl_sync(0xffffffffu, bq, base | 2);
                    const float b3 = __shfl_sync(0xffffffffu, bq, base | 3);
                    const float v0 = b0;
                    const float v1 = fmaf(d10, b0, b1);
                    const float v2 = fmaf(d21, b1, fmaf(d20, b0, b2));
                    const float v3 = fmaf(d32, b2, fmaf(d31, b1, fmaf(d30, b0, b3)));
                    p[tau] = q == 0 ? v0 : (q == 1 ? v1 : (q == 2 ? v2 : v3));
#pragma unroll
                    for (int m = tau + 1; m < 16; ++m) {
                        const float4 am = *reinterpret_cast<const float4 *>(Af + (4 * m + q) * wy::kAs + 4 * tau);
                        p[m] = fmaf(am.w, v3, fmaf(am.z, v2, fmaf(am.y, v1, fmaf(am.x, v0, p[m]))));
                    }
                }
            }
            if (warp >= 4) {
                // The warps with few pivot steps (column blocks 4..7) then
                // write the dec o K parts for the scan's state update, an
                // MN-major operand with the K rows' layout (64-column atoms
                // 8 KB apart): 16-byte piece e of the output (atom e/512,
                // token row i) is the same piece of A1's K row i, scaled by dec_i.
                for (int e = tid - 128; e < kD * kC / 8; e += kThreads - 128) {
                    const int atom = e >> 9, i = (e >> 3) & (kC - 1);
                    const uint4 kr = *reinterpret_cast<const uint4 *>(sm + wy::kA1 + atom * 16384 + (e & 511) * 16);
                    const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w};
                    const float di = dec[i];
                    float kv[8];
#pragma unroll
                    for (int y = 0; y < 8; ++y)
                        kv[y] = gdn::bf16_to_f32(uint16_t(y & 1 ? kw[y >> 1] >> 16 : kw[y >> 1] & 0xffffu)) * di;
                    uint4 hi, lo;
                    split8(kv, hi, lo);
                    *reinterpret_cast<uint4 *>(out + blob::kK1 + e * 16) = hi;
                    *reinterpret_cast<uint4 *>(out + blob::kK2 + e * 16) = lo;
                }
            }
            __syncthreads();  // every A entry is read before T overwrites it
#pragma unroll
            for (int m = 0; m < 16; ++m) Af[(4 * m + q) * wy::kAs + j] = p[m];
        }
        __syncthreads();
        // AB rows t: T diag(beta e^G); rows 64 + t: T diag(beta); hi and lo parts.
        const int t = tid >> 2, i0 = (tid & 3) * 16;
        float tv[16];
#pragma unroll
        for (int x = 0; x < 16; x += 4) {
            const float4 tr = *reinterpret_cast<const float4 *>(Af + t * wy::kAs + i0 + x);
            tv[x] = tr.x;
            tv[x + 1] = tr.y;
            tv[x + 2] = tr.z;
            tv[x + 3] = tr.w;
        }
        __syncthreads();  // every T entry is read before the tiles overwrite it
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float xb[8], xv[8];
#pragma unroll
            for (int y = 0; y < 8; ++y) {
                const int i = i0 + half * 8 + y;
                xv[y] = tv[half * 8 + y] * Bs[i];
                xb[y] = xv[y] * eG[i];
            }
            uint4 bh, bl, vh, vl;
            split8(xb, bh, bl);
            split8(xv, vh, vl);
            const uint32_t ob = tc::swz_off(128, t, i0 + half * 8), ov = tc::swz_off(128, kC + t, i0 + half * 8);
            *reinterpret_cast<uint4 *>(sm + wy::kAbHi + ob) = bh;
            *reinterpret_cast<uint4 *>(sm + wy::kAbLo + ob) = bl;
            *reinterpret_cast<uint4 *>(sm + wy::kAbHi + ov) = vh;
            *reinterpret_cast<uint4 *>(sm + wy::kAbLo + ov) = vl;
        }
        gdn::fence_proxy_async_smem();
        tc::fence_before();
    }
    __syncthreads();
    if (ok && tid == 0) {
        tc::fence_after();
        // D2 = AB [K | V] (M = 128, N = 256, B MN-major: four 64-column
        // blocks 16 KB apart from A1's K rows to VN); hi and lo parts accumulate.
        constexpr uint32_t idesc = tc::idesc_bf16(128, 256) | tc::kBMnMajor;
        const uint64_t bkv = tc::smem_desc_mn(sb + wy::kA1, 16384);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const uint64_t b = tc::desc_at(bkv, s * 2048);
            tc::mma_bf16(tm, tc::smem_desc(sb + wy::kAbHi + s * 32), b, idesc, s ? 1u : 0u);
            tc::mma_bf16(tm, tc::smem_desc(sb + wy::kAbLo + s * 32), b, idesc, 1u);
        }
        tc::commit(bar);
        *flag = gdn::mbar_wait_bounded(bar, 1) ? 1 : 0;
    }
    __syncthreads();
    ok = ok && *flag != 0;
    if (ok) {
        (void)gdn::mbar_try_wait(bar, 1);
        tc::fence_after();
        const int q4 = warp & 3, hc = warp >> 2;
        const int t = 32 * (q4 & 1) + lane;  // token row = accumulator lane (mod 64)
        const uint32_t lane_base = uint32_t(32 * q4) << 16;
        if (q4 < 2) {
            // W row t -> its two bf16 parts (columns 64hc.. in atom hc)
#pragma unroll
            for (int part = 0; part < 4; ++part) {
                const int col = 16 * part;
                float w16[16];
                tc::ld16(tm + lane_base + uint32_t(64 * hc + col), w16);
#pragma unroll
                for (int x = 0; x < 16; x += 8) {
                    uint4 hi, lo;
                    split8(w16 + x, hi, lo);
                    const uint32_t off = tc::swz_off(64, t, col + x);
                    *reinterpret_cast<uint4 *>(sm + wy::st_w1(hc) + off) = hi;
                    *reinterpret_cast<uint4 *>(sm + wy::st_w2(hc) + off) = lo;
                }
            }
        } else {
            // Ut row t, fp32, staged where AB was
            float *Ut = reinterpret_cast<float *>(sm + wy::kStUt);
#pragma unroll
            for (int part = 0; part < 4; ++part) {
                const int col = 64 * hc + 16 * part;
                float u16[16];
                tc::ld16(tm + lane_base + 128u + uint32_t(col), u16);
#pragma unroll
                for (int x = 0; x < 16; x += 4)
                    *reinterpret_cast<float4 *>(Ut + ut_index(t, col + x)) =
                        make_float4(u16[x], u16[x + 1], u16[x + 2], u16[x + 3]);
            }
        }
        gdn::fence_proxy_async_smem();
    } else if (tid == 0) {
        gdn::set_status(a.status, GDN_DEV_TIMEOUT);
    }
    tc::fence_before();
    __syncthreads();
    if (tid == 0) {
        if (ok) {
            // W and Ut parts.
            for (int at = 0; at < 2; ++at) {
                gdn::bulk_s2g(out + blob::kW1Q + at * 16384, sm + wy::st_w1(at), 8192u);
                gdn::bulk_s2g(out + blob::kW2 + at * 8192, sm + wy::st_w2(at), 8192u);
            }
            gdn::bulk_s2g(out + blob::kUt, sm + wy::kStUt, 16384u);
            gdn::bulk_s2g(out + blob::kUt + 16384, sm + wy::kStUt + 16384, 16384u);
            gdn::bulk_commit();
        }
        // The stores have read their shared-memory sources before it is
        // released; their writes are complete when the grid is.
        gdn::bulk_wait_read_all();
    }
    if (warp == 0) tc::tmem_dealloc(tm, wy::kTmemCols);
}

// ---------------------------------------------------------------------------
// (2) sequential scan over chunks on the tensor cores (tcgen05, kind::f16)
// ---------------------------------------------------------------------------
// One CTA per (sequence, v-head); the 128 value rows of S are the M = 128
// side of every product, so each thread owns one row of S (lane quadrant of
// its warp) and a quarter of its columns (16 warps).  The FP32 master copy of S stays in
// registers for the whole sequence.  S and U are split into two bf16 parts
// here; W, P and dec o K arrive split from the per-chunk kernel; a product
// keeps the three leading terms a1 b1 + a1 b2 + a2 b1; q and k are exact
// bf16.  Per chunk:
//   phase A:  Uacc = S W^T         (M128 N64  K128)  -> U^T = Ut^T - Uacc
//             Oi   = S Q^T         (M128 N64  K128)
//   phase B:  Oa   = U^T P^T       (M128 N64  K64)
//             dS   = U^T (dec o K) (M128 N128 K64),   S <- e^{G_last} S + dS
//   o_t = q_scale (e^{G_t} Oi[:,t] + Oa[:,t]),  dec_i = e^{G_last - G_i}.
// Shared-memory map (bytes from a 1024-aligned base), bf16 K-major tiles:
namespace sc {
constexpr uint32_t kS1 = 0, kS2 = 32768;  // S parts       128 rows (d_v) x 128 (d_k)
constexpr uint32_t kTiles = 65536;        // the chunk's W, Q, P and dec o K tiles, in the workspace layout
constexpr uint32_t kW1Q = kTiles + blob::kW1Q, kW2 = kTiles + blob::kW2;
constexpr uint32_t kP1 = kTiles + blob::kP1, kP2 = kTiles + blob::kP2;
constexpr uint32_t kK1 = kTiles + blob::kK1, kK2 = kTiles + blob::kK2;
constexpr uint32_t kU1 = kTiles + blob::kTiles, kU2 = kU1 + 16384;  // U^T parts 128 rows (d_v) x 64 (i)
constexpr uint32_t kMisc = kU2 + 16384;   // e^G (two chunks' worth), mbarriers, tensor-memory base, flag
constexpr size_t kSmem = kMisc + 1024 + 1024;
constexpr uint32_t kTmemCols = 512;  // Uacc 0..63, dS 256..383, Oi/Oa two buffers
}  // namespace sc

// Fetches of chunk c's workspace blob, issued by one thread: part A (the W
// and Q tiles, 48 KB) is needed by the chunk's first products and may land
// once the previous chunk's first products are done; part B (P and dec o K,
// 48 KB, and e^G into buffer c % 2) is needed from the second products on.
__device__ __forceinline__ void scan_fetch_a(const PrefArgs &a, unsigned char *sm, uint64_t *bar, int s0, int seq,
                                             int h, int c) {
    const unsigned char *src = ws_blob(a, chunk_slot(s0, c, seq), h);
    gdn::fence_proxy_async_smem();
    gdn::mbar_arrive_expect_tx(bar, 3u * 16384u);
    for (int i = 0; i < 3; ++i) gdn::bulk_g2s(sm + sc::kTiles + i * 16384, src + i * 16384, 16384u, bar);
}
__device__ __forceinline__ void scan_fetch_b(const PrefArgs &a, unsigned char *sm, uint64_t *bar, int s0, int seq,
                                             int h, int c) {
    const unsigned char *src = ws_blob(a, chunk_slot(s0, c, seq), h);
    gdn::fence_proxy_async_smem();
    gdn::mbar_arrive_expect_tx(bar, 3u * 16384u + 256u);
    for (int i = 3; i < 6; ++i) gdn::bulk_g2s(sm + sc::kTiles + i * 16384, src + i * 16384, 16384u, bar);
    gdn::bulk_g2s(sm + sc::kMisc + (c & 1) * 256, src + blob::kEG, 256u, bar);
}

__global__ void __launch_bounds__(kScanThreads, 1) gdn_chunk_scan_kernel(const PrefArgs a) {
    const int h = blockIdx.x % a.h_v;
    const int seq = a.order[blockIdx.x / a.h_v];  // longest sequences start first
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

    extern __shared__ unsigned char smraw[];
    const uint32_t raw_u = gdn::smem_u32(smraw);
    unsigned char *sm = smraw + (((raw_u + 1023u) & ~1023u) - raw_u);
    const uint32_t sb = gdn::smem_u32(sm);
    uint64_t *bar_u = reinterpret_cast<uint64_t *>(sm + sc::kMisc + 768);   // Uacc done
    uint64_t *bar_ia = reinterpret_cast<uint64_t *>(sm + sc::kMisc + 784);  // W, Q tiles arrived
    uint64_t *bar_b = reinterpret_cast<uint64_t *>(sm + sc::kMisc + 792);   // phase B done
    uint64_t *bar_o = reinterpret_cast<uint64_t *>(sm + sc::kMisc + 800);   // Oi done
    uint64_t *bar_ib = reinterpret_cast<uint64_t *>(sm + sc::kMisc + 808);  // P, dec o K, e^G arrived
    uint32_t *tbase = reinterpret_cast<uint32_t *>(sm + sc::kMisc + 776);
    int *flag = reinterpret_cast<int *>(sm + sc::kMisc + 780);
    int *oflag = reinterpret_cast<int *>(sm + sc::kMisc + 816);  // the Oi wait of the fetching thread

    if (warp == 0) tc::tmem_alloc(tbase, sc::kTmemCols);
    if (tid == 0) {
        gdn::mbar_init(bar_u, 1);
        gdn::mbar_init(bar_ia, 1);
        gdn::mbar_init(bar_b, 1);
        gdn::mbar_init(bar_o, 1);
        gdn::mbar_init(bar_ib, 1);
    }

    const int q4 = warp & 3, cq = warp >> 2;  // lane quadrant, column quarter
    const int arow = 32 * q4 + lane;          // row of S held by this thread
    const uint32_t lane_base = uint32_t(32 * q4) << 16;
    const size_t row_off = size_t(h) * kD * kD + size_t(arow) * kD + 32 * cq;
    float sv[32];  // S[arow][32cq .. 32cq+31], FP32 master
    if (src >= 0) {
        const float4 *sp = reinterpret_cast<const float4 *>(a.pool + size_t(src) * a.slot_stride + row_off);
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            const float4 v = sp[x];
            sv[4 * x] = v.x;
            sv[4 * x + 1] = v.y;
            sv[4 * x + 2] = v.z;
            sv[4 * x + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int x = 0; x < 32; ++x) sv[x] = 0.f;
    }
    auto write_S = [&]() {
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            uint4 hi, lo;
            split8(sv + 8 * x, hi, lo);
            const uint32_t off = tc::swz_off(128, arow, 32 * cq + 8 * x);
            *reinterpret_cast<uint4 *>(sm + sc::kS1 + off) = hi;
            *reinterpret_cast<uint4 *>(sm + sc::kS2 + off) = lo;
        }
        gdn::fence_proxy_async_smem();
        tc::fence_before();
    };
    write_S();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tbase;
    constexpr uint32_t id64 = tc::idesc_bf16(128, 64);
    constexpr uint32_t id128 = tc::idesc_bf16(128, 128);
    // Tensor-memory columns: dS 256..383, and for chunk c in buffer c % 2
    // [Uacc | Oi] (128 columns) and Oa (the outputs of chunk c are read while
    // chunk c + 1's first products run): buffer 0 at 0..127 and 128..191,
    // buffer 1 at 384..511 and 192..255.
    const uint64_t dsc = tc::smem_desc(sb);  // descriptors of the fixed tiles: tc::desc_at(dsc, offset)
    const uint64_t dsc_k = tc::smem_desc_mn(sb + sc::kK1, 8192);  // dec o K parts, MN-major B (K2 at +16 KB)
    constexpr uint32_t id128k = id128 | tc::kBMnMajor;
    auto uo_col = [](int b) { return uint32_t(384 * b); };  // Uacc at +0, Oi at +64
    auto oi_col = [](int b) { return uint32_t(384 * b + 64); };
    auto oa_col = [](int b) { return uint32_t(128 + 64 * b); };
    // Phase A of chunk c (thread 0): [Uacc | Oi] = S [W1; Q]^T (N = 128) for
    // both parts of S, plus S1 W2^T into Uacc (N = 64); committed to bar_u and
    // bar_o (W and Q are then free for the next chunk's fetch).
    auto issue_phase_a = [&](int c) {
        tc::fence_after();
        const uint32_t d = tm + uo_col(c & 1);
#pragma unroll
        for (int at = 0; at < 2; ++at)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint32_t ka = at * 16384 + s * 32;
                const uint64_t a1 = tc::desc_at(dsc, sc::kS1 + ka), a2 = tc::desc_at(dsc, sc::kS2 + ka);
                const uint64_t wq = tc::desc_at(dsc, sc::kW1Q + ka);
                const uint64_t w2 = tc::desc_at(dsc, sc::kW2 + at * 8192 + s * 32);
                tc::mma_bf16(d, a1, wq, id128, (at | s) ? 1u : 0u);
                tc::mma_bf16(d, a1, w2, id64, 1u);
                tc::mma_bf16(d, a2, wq, id128, 1u);
            }
        tc::commit(bar_u);
        tc::commit(bar_o);
    };
    // Per-thread Ut values of chunk c: Ut[t][arow] for t in [16cq, 16cq+16).
    float ut[16];
    auto load_ut = [&](int c) {
        const float *Ut = reinterpret_cast<const float *>(ws_blob(a, chunk_slot(s0, c, seq), h) + blob::kUt);
#pragma unroll
        for (int x = 0; x < 16; ++x) ut[x] = Ut[ut_index(16 * cq + x, arow)];
    };

    // Outputs of chunk c: o_t = q_scale (e^{G_t} Oi[:,t] + Oa[:,t]) for the
    // 16 tokens of this thread's column quarter.  They are written one chunk
    // late, while the next chunk's phase B runs (the other warps wait for it
    // anyway); thread 0 is then issuing that phase, so the columns of warp 0
    // (tokens 0..15 of lane quadrant 0) go to warps 4 and 8, eight each.
    auto outputs_part = [&](int c, int col0, int x0, int x1) {
        const int t0 = s0 + c * kC;
        const int n = min(kC, len - c * kC);
        const float *eG = reinterpret_cast<const float *>(sm + sc::kMisc + (c & 1) * 256);
        float oi[16], oa[16];
        tc::ld16(tm + lane_base + oi_col(c & 1) + uint32_t(col0), oi);
        tc::ld16(tm + lane_base + oa_col(c & 1) + uint32_t(col0), oa);
#pragma unroll
        for (int x = 0; x < 16; ++x) {
            const int t = col0 + x;
            if (x >= x0 && x < x1 && t < n)
                a.o[(size_t(t0 + t) * a.h_v + h) * kD + arow] =
                    gdn::f32_to_bf16(a.q_scale * fmaf(eG[t], oi[x], oa[x]));
        }
    };
    auto write_outputs = [&](int c) {
        if (warp != 0) outputs_part(c, 16 * cq, 0, 16);
        if (warp == 4) outputs_part(c, 0, 0, 8);
        if (warp == 8) outputs_part(c, 0, 8, 16);
    };

    uint32_t par_u = 0, par_b = 0, par_o = 0, par_ia = 0, par_ib = 0;
    bool ok = true;
    const int nchunks = (len + kC - 1) / kC;
    if (nchunks > 0) {
        load_ut(0);
        if (tid == 0) {
            scan_fetch_a(a, sm, bar_ia, s0, seq, h, 0);
            scan_fetch_b(a, sm, bar_ib, s0, seq, h, 0);
            const bool got = gdn::mbar_wait_bounded(bar_ia, par_ia);
            *flag = got ? 1 : 0;
            if (got) issue_phase_a(0);
        }
        par_ia ^= 1u;
        __syncthreads();
        ok = *flag != 0;
    }
    for (int c = 0; ok && c < nchunks; ++c) {
        const int t0 = s0 + c * kC;
        const int n = min(kC, len - c * kC);
        const bool more = c + 1 < nchunks;
        const float *eG = reinterpret_cast<const float *>(sm + sc::kMisc + (c & 1) * 256);
        // Uacc of this chunk.
        if (tid == 0) *flag = gdn::mbar_wait_bounded(bar_u, par_u) ? 1 : 0;
        par_u ^= 1u;
        __syncthreads();
        if (*flag == 0) {
            ok = false;
            break;
        }
        tc::fence_after();
        // The next chunk's W and Q can land as soon as this chunk's Oi product
        // is done with W and Q: a second thread waits for it and starts the
        // fetch while the U split and phase B run.
        if (tid == 32) {
            const bool got = gdn::mbar_wait_bounded(bar_o, par_o);
            *oflag = got ? 1 : 0;
            if (got && more) scan_fetch_a(a, sm, bar_ia, s0, seq, h, c + 1);
        }
        par_o ^= 1u;
        // U^T[arow][t] = Ut[t][arow] - Uacc[arow][t], split into two bf16 parts.
        {
            float v16[16];
            const int col0 = 16 * cq;
            tc::ld16(tm + lane_base + uo_col(c & 1) + uint32_t(col0), v16);
#pragma unroll
            for (int x = 0; x < 16; x += 8) {
                float u[8];
#pragma unroll
                for (int y = 0; y < 8; ++y) u[y] = ut[x + y] - v16[x + y];
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
        // Phase B: Oa = U^T P^T, dS = U^T (dec o K), once this chunk's P and
        // dec o K have arrived; meanwhile the next chunk's W and Q are fetched
        // as soon as this chunk's Oi is done with W and Q.
        bool good_b = true;
        if (tid == 0) {
            bool good = gdn::mbar_wait_bounded(bar_ib, par_ib);
            if (good) {
                tc::fence_after();
                const uint32_t oa = tm + oa_col(c & 1);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t u1 = tc::desc_at(dsc, sc::kU1 + s * 32), u2 = tc::desc_at(dsc, sc::kU2 + s * 32);
                    const uint64_t p1 = tc::desc_at(dsc, sc::kP1 + s * 32), p2 = tc::desc_at(dsc, sc::kP2 + s * 32);
                    const uint64_t k1 = tc::desc_at(dsc_k, s * 2048), k2 = tc::desc_at(dsc_k, (sc::kK2 - sc::kK1) + s * 2048);
                    tc::mma_bf16(oa, u1, p1, id64, s ? 1u : 0u);
                    tc::mma_bf16(oa, u1, p2, id64, 1u);
                    tc::mma_bf16(oa, u2, p1, id64, 1u);
                    tc::mma_bf16(tm + 256, u1, k1, id128k, s ? 1u : 0u);
                    tc::mma_bf16(tm + 256, u1, k2, id128k, 1u);
                    tc::mma_bf16(tm + 256, u2, k1, id128k, 1u);
                }
                tc::commit(bar_b);
            }
            good_b = good;
        }
        if (c > 0) write_outputs(c - 1);  // while phase B runs
        if (tid == 0) {
            const bool good = good_b && gdn::mbar_wait_bounded(bar_b, par_b);
            *flag = (good && *oflag) ? 1 : 0;
        }
        par_ib ^= 1u;
        par_b ^= 1u;
        __syncthreads();
        if (*flag == 0) {
            ok = false;
            break;
        }
        tc::fence_after();
        // Every product of this chunk is done: P and dec o K are free for the next chunk's.
        if (more && tid == 0) scan_fetch_b(a, sm, bar_ib, s0, seq, h, c + 1);
        // S <- e^{G_last} S + dS (FP32 master), then its bf16 parts.
        const float egl = eG[n - 1];
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            float v16[16];
            tc::ld16(tm + lane_base + 256u + uint32_t(32 * cq + 16 * part), v16);
#pragma unroll
            for (int x = 0; x < 16; ++x) sv[16 * part + x] = fmaf(egl, sv[16 * part + x], v16[x]);
        }
        write_S();
        if (more) {
            load_ut(c + 1);
            if (tid == 0) *flag = gdn::mbar_wait_bounded(bar_ia, par_ia) ? 1 : 0;
            par_ia ^= 1u;
            __syncthreads();  // the S parts are written and the next chunk's W and Q have arrived
            if (*flag == 0) {
                ok = false;
                break;
            }
            if (tid == 0) issue_phase_a(c + 1);
        }
        tc::fence_before();
    }
    if (ok && nchunks > 0) {
        tc::fence_after();
        write_outputs(nchunks - 1);
    }
    if (ok) {
        float4 *dp = reinterpret_cast<float4 *>(a.pool + size_t(dst) * a.slot_stride + row_off);
#pragma unroll
        for (int x = 0; x < 8; ++x) dp[x] = make_float4(sv[4 * x], sv[4 * x + 1], sv[4 * x + 2], sv[4 * x + 3]);
    } else if (tid == 0) {
        gdn::set_status(a.status, GDN_DEV_TIMEOUT);
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, sc::kTmemCols);
}

// order[r] = the sequence with the r-th largest length (ties by index), so
// that the scan's longest dependency chains are scheduled in its first wave;
// chunk_seq[x] = the sequence whose chunk sits in workspace slot x (-1 for
// none), so that the per-chunk kernel's grid covers only the slot range.
// One block: sequences that fail the scan's row checks get no chunks.
__global__ void gdn_prefill_tables_kernel(const int32_t *cu, int nseq, int row_capacity, int nslots,
                                          int32_t *order, int32_t *chunk_seq) {
    for (int x = threadIdx.x; x < nslots; x += blockDim.x) chunk_seq[x] = -1;
    for (int i = threadIdx.x; i < nseq; i += blockDim.x) {
        const int li = cu[i + 1] - cu[i];
        int r = 0;
        for (int j = 0; j < nseq; ++j) {
            const int lj = cu[j + 1] - cu[j];
            r += (lj > li || (lj == li && j < i)) ? 1 : 0;
        }
        order[r] = i;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    for (int i = warp; i < nseq; i += nwarps) {
        const int s0 = cu[i], s1 = cu[i + 1];
        if (s0 < 0 || s1 < s0 || s1 > row_capacity) continue;
        const int nch = (s1 - s0 + kC - 1) / kC;
        for (int c = lane; c < nch; c += 32) chunk_seq[chunk_slot(s0, c, i)] = i;
    }
}

constexpr size_t kWySmem = wy::kSmem;
constexpr size_t kScanSmem = sc::kSmem;

}  // namespace

// Chunk slots: sequence i's chunk c uses slot chunk_slot(cu[i], c, i), which
// is below ceil(row_capacity / 64) + nseq for every valid sequence.
static size_t chunk_slots(int32_t nseq, int32_t row_capacity) {
    return size_t((int64_t(row_capacity) + kC - 1) / kC) + size_t(nseq);
}

static size_t blobs_bytes(const gdn_dims *dims, int32_t nseq, int32_t row_capacity) {
    return chunk_slots(nseq, row_capacity) * size_t(dims->h_v) * kWsFloats * sizeof(float);
}

static size_t align16(size_t x) { return (x + 15) / 16 * 16; }

// cuTensorMapEncodeTiled, reached through the runtime's driver entry points.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// Rows of `heads` x 128 bf16 values (rows x heads x 128, innermost last) as a
// 3-D tensor with boxes of 64 values x 1 head x 64 rows, 128-byte swizzled.
static bool encode_rows(CUtensorMap *m, const void *base, int heads, int rows) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[3] = {cuuint64_t(kD), cuuint64_t(heads), cuuint64_t(rows > 0 ? rows : 1)};
    const cuuint64_t strides[2] = {cuuint64_t(kD) * 2, cuuint64_t(heads) * kD * 2};
    const cuuint32_t box[3] = {64, 1, kC};
    const cuuint32_t elem[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Workspace: the blobs, then order[nseq], then chunk_seq[slots].
extern "C" size_t gdn_prefill_workspace_bytes(const gdn_dims *dims, int32_t nseq, int32_t row_capacity) {
    if (!dims || nseq < 0 || row_capacity < 0) return 0;
    return blobs_bytes(dims, nseq, row_capacity) + align16(size_t(nseq) * 4) +
           align16(chunk_slots(nseq, row_capacity) * 4);
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
    if (!gdn_host::aligned16(workspace)) return GDN_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    PrefArgs a{};
    a.cu = cu_seqlens;
    a.nseq = nseq;
    a.h_qk = dims->h_qk;
    a.h_v = dims->h_v;
    a.grp = dims->h_v / dims->h_qk;
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
    unsigned char *tables = static_cast<unsigned char *>(workspace) + blobs_bytes(dims, nseq, row_capacity);
    int32_t *order = reinterpret_cast<int32_t *>(tables);
    int32_t *chunk_seq = reinterpret_cast<int32_t *>(tables + align16(size_t(nseq) * 4));
    a.order = order;
    a.chunk_seq = chunk_seq;
    a.q_scale = dims->q_scale;
    a.status = dev_status;
    if (!encode_rows(&a.tm_q, q, dims->h_qk, row_capacity) || !encode_rows(&a.tm_k, k, dims->h_qk, row_capacity) ||
        !encode_rows(&a.tm_v, v, dims->h_v, row_capacity))
        return GDN_ERR_CUDA;
    if (cudaFuncSetAttribute(gdn_chunk_wy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kWySmem)) !=
            cudaSuccess ||
        cudaFuncSetAttribute(gdn_chunk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kScanSmem)) !=
            cudaSuccess)
        return GDN_ERR_CUDA;
    const size_t slots = chunk_slots(nseq, row_capacity);
    if (slots > 0x7fffffffULL || dims->h_v > 65535) return GDN_ERR_ARG;
    gdn_prefill_tables_kernel<<<1, 1024, 0, st>>>(cu_seqlens, nseq, row_capacity, int(slots), order, chunk_seq);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    gdn_chunk_wy_kernel<<<dim3(unsigned(slots), dims->h_v), kThreads, kWySmem, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    const long long gs = (long long)nseq * dims->h_v;
    gdn_chunk_scan_kernel<<<unsigned(gs), kScanThreads, kScanSmem, st>>>(a);
    return gdn_host::launch_status(cudaGetLastError());
}
