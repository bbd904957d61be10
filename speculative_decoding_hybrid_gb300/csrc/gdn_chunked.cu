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
// (1) per-chunk WY/UT quantities
// ---------------------------------------------------------------------------
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

    extern __shared__ __align__(16) float sm[];
    float *Ks = sm;                    // [C][D+1]
    float *Vs = Ks + kC * (kD + 1);    // [C][D+1]
    float *Ts = Vs + kC * (kD + 1);    // [C][C+1]  A, then T
    float *Gs = Ts + kC * (kC + 1);    // [C]
    float *Bs = Gs + kC;               // [C]
    const int tid = threadIdx.x;

    for (int i = tid; i < kC * kD; i += kThreads) {
        const int t = i / kD, j = i % kD;
        float kv = 0.f, vv = 0.f;
        if (t < n) {
            kv = gdn::bf16_to_f32(a.k[(size_t(t0 + t) * a.h_qk + hq) * kD + j]);
            vv = gdn::bf16_to_f32(a.v[(size_t(t0 + t) * a.h_v + h) * kD + j]);
        }
        Ks[t * (kD + 1) + j] = kv;
        Vs[t * (kD + 1) + j] = vv;
    }
    if (tid < kC) {
        Bs[tid] = tid < n ? a.beta[size_t(t0 + tid) * a.h_v + h] : 0.f;
        Gs[tid] = tid < n ? a.g[size_t(t0 + tid) * a.h_v + h] : 0.f;
    }
    __syncthreads();
    if (tid == 0) {  // G = cumsum(g) within the chunk
        float run = 0.f;
        for (int t = 0; t < kC; ++t) {
            run += Gs[t];
            Gs[t] = run;
        }
    }
    __syncthreads();
    // A[t][i] = beta_t e^{G_t-G_i} k_t.k_i for i < t (16 entries per thread)
    for (int e = tid; e < kC * kC; e += kThreads) {
        const int t = e / kC, i = e % kC;
        float val = 0.f;
        if (i < t && t < n) {
            float acc = 0.f;
            for (int j = 0; j < kD; ++j) acc = fmaf(Ks[t * (kD + 1) + j], Ks[i * (kD + 1) + j], acc);
            val = Bs[t] * expf(Gs[t] - Gs[i]) * acc;
        }
        Ts[t * (kC + 1) + i] = val;
    }
    __syncthreads();
    // T = (I + A)^{-1}: column i of T depends only on column i of earlier rows,
    // so thread i substitutes its column alone (A in the strict lower part,
    // T written over it row by row: T[t][i] needs A[t][m] for m >= i only).
    float col[kC];
    if (tid < kC) {
        const int i = tid;
        for (int t = 0; t < kC; ++t) col[t] = 0.f;
        col[i] = 1.f;
        for (int t = i + 1; t < kC; ++t) {
            float acc = 0.f;
            for (int m = i; m < t; ++m) acc = fmaf(Ts[t * (kC + 1) + m], col[m], acc);
            col[t] = -acc;
        }
    }
    __syncthreads();  // every column has read A before any is overwritten
    if (tid < kC)
        for (int t = 0; t < kC; ++t) Ts[t * (kC + 1) + tid] = col[t];
    __syncthreads();
    // W[t][j] = sum_i T[t][i] beta_i e^{G_i} K[i][j],  Ut[t][a] = sum_i T[t][i] beta_i V[i][a]
    float *W = ws_w(a, chunk_slot(s0, c, seq), h);
    float *Ut = W + kC * kD;
    for (int e = tid; e < kC * kD; e += kThreads) {
        const int t = e / kD, j = e % kD;
        float aw = 0.f, au = 0.f;
        for (int i = 0; i <= t; ++i) {
            const float tb = Ts[t * (kC + 1) + i] * Bs[i];
            aw = fmaf(tb * expf(Gs[i]), Ks[i * (kD + 1) + j], aw);
            au = fmaf(tb, Vs[i * (kD + 1) + j], au);
        }
        W[e] = aw;
        Ut[e] = au;
    }
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

constexpr size_t kWySmem = sizeof(float) * (2 * kC * (kD + 1) + kC * (kC + 1) + 2 * kC);
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
