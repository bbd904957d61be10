// Chunked (WY/UT) GatedDeltaNet prefill for d_k = d_v in {16, 32, 64}, in
// plain fp32 on the CUDA cores (sm_103a).
//
// "Run chained MTP drafting in the batch Engine", Correctness fix: the
// chunked plan runs a whole prompt at once and publishes only its final
// state; it must take every prompt the recurrent plan takes, including the
// smaller head sizes the recurrent kernels serve.  Per chunk of C = 64
// tokens (n of them valid) with start state S (d_v x d_k) and G = cumsum(g):
//   A[t][i] = beta_t e^{G_t-G_i} k_t.k_i  (i < t),   T = (I + A)^{-1}
//   W  = T diag(beta e^G) K,   Ut = T diag(beta) V,   U = Ut - W S^T
//   O  = diag(e^G) Q S^T + P U,   P[t][i] = e^{G_t-G_i} q_t.k_i  (i <= t)
//   S' = e^{G_last} S + U^T diag(dec) K,   dec_i = e^{G_last-G_i}
// At these sizes a 128-row tensor-core tile would be mostly padding, so one
// CTA of 256 threads per (sequence, v-head) runs the chunk form in fp32 in
// shared memory, walking the sequence's chunks.  Nothing is written but the
// outputs and the final state.
#include "chunk_math.cuh"

namespace {

constexpr int kC = 64;
constexpr int kThreads = 256;
constexpr int kAs = 68;  // row stride (floats) of the 64 x 64 matrices

template <int D>
struct SmallLay {
    static constexpr int Ds = D + 1;  // padded row stride of the d-wide rows
    static constexpr size_t kS = 0;                                   // S [D][Ds]
    static constexpr size_t kK = kS + size_t(D) * Ds;                 // K [64][Ds]
    static constexpr size_t kQ = kK + size_t(kC) * Ds;                // Q
    static constexpr size_t kV = kQ + size_t(kC) * Ds;                // V
    static constexpr size_t kW = kV + size_t(kC) * Ds;                // W
    static constexpr size_t kU = kW + size_t(kC) * Ds;                // Ut, then U
    static constexpr size_t kA = (kU + size_t(kC) * Ds + 3) / 4 * 4;  // A -> T [64][kAs] (16-byte rows)
    static constexpr size_t kP = kA + size_t(kC) * kAs;               // P [64][kAs]
    static constexpr size_t kX = kP + size_t(kC) * kAs;               // solve scratch (32 x 36)
    static constexpr size_t kVec = kX + 32 * 36;                      // G, e^G, dec, beta (64 each)
    static constexpr size_t kFloats = kVec + 4 * kC;
    static constexpr size_t kBytes = kFloats * 4;
};

struct SmallArgs {
    const int32_t *cu;
    int32_t h_qk, h_v, grp, row_capacity, num_slots;
    const uint16_t *q, *k, *v;
    const float *g, *beta;
    float *pool;
    int64_t slot_stride;
    const int32_t *src_slot, *dst_slot;
    uint16_t *o;
    const int32_t *order;
    float q_scale;
    uint32_t *status;
};

template <int D>
__global__ void __launch_bounds__(kThreads) gdn_prefill_small_kernel(const SmallArgs a) {
    using L = SmallLay<D>;
    constexpr int Ds = L::Ds;
    const int h = blockIdx.x % a.h_v;
    const int seq = a.order[blockIdx.x / a.h_v];
    const int tid = threadIdx.x;
    const int s0 = a.cu[seq], s1 = a.cu[seq + 1], len = s1 - s0;
    const int src = a.src_slot[seq], dst = a.dst_slot[seq];
    uint32_t bad = 0;
    if (s0 < 0 || len < 0 || s1 > a.row_capacity) bad |= GDN_DEV_ROWS_BAD;
    if (src < -1 || src >= a.num_slots || dst < 0 || dst >= a.num_slots) bad |= GDN_DEV_SLOT_OOR;
    if (bad) {
        if (h == 0 && tid == 0) gdn::set_status(a.status, bad);
        return;
    }
    const int hq = h / a.grp;
    extern __shared__ __align__(16) float smf[];
    float *S = smf + L::kS, *K = smf + L::kK, *Q = smf + L::kQ, *V = smf + L::kV;
    float *W = smf + L::kW, *U = smf + L::kU, *Af = smf + L::kA, *P = smf + L::kP, *X = smf + L::kX;
    float *G = smf + L::kVec, *eG = G + kC, *dec = eG + kC, *Bt = dec + kC;
    const size_t head_off = size_t(h) * D * D;
    for (int e = tid; e < D * D; e += kThreads)
        S[(e / D) * Ds + e % D] = src >= 0 ? a.pool[size_t(src) * a.slot_stride + head_off + e] : 0.f;

    const int nch = (len + kC - 1) / kC;
    for (int c = 0; c < nch; ++c) {
        const int t0 = s0 + c * kC, n = min(kC, len - c * kC);
        // the chunk's rows in fp32 (zero past its n tokens), its gates
        for (int e = tid; e < kC * D; e += kThreads) {
            const int t = e / D, j = e % D;
            float kv = 0.f, qv = 0.f, vv = 0.f;
            if (t < n) {
                kv = gdn::bf16_to_f32(a.k[(size_t(t0 + t) * a.h_qk + hq) * D + j]);
                qv = gdn::bf16_to_f32(a.q[(size_t(t0 + t) * a.h_qk + hq) * D + j]);
                vv = gdn::bf16_to_f32(a.v[(size_t(t0 + t) * a.h_v + h) * D + j]);
            }
            K[t * Ds + j] = kv;
            Q[t * Ds + j] = qv;
            V[t * Ds + j] = vv;
        }
        if (tid < kC) {
            G[tid] = tid < n ? a.g[size_t(t0 + tid) * a.h_v + h] : 0.f;
            Bt[tid] = tid < n ? a.beta[size_t(t0 + tid) * a.h_v + h] : 0.f;
        }
        __syncthreads();
        if (tid < 32) {
            chunkmath::chunk_cumsum(G, n, G);
            __syncwarp();
            const float gl = G[n - 1];
            for (int e = tid; e < kC; e += 32) {
                eG[e] = expf(G[e]);
                dec[e] = e < n ? expf(gl - G[e]) : 0.f;
            }
        }
        __syncthreads();
        // A and P: 64 x 64 entries each, d-long dot products
        for (int e = tid; e < kC * kC; e += kThreads) {
            const int t = e / kC, i = e % kC;
            float kk = 0.f, qk = 0.f;
#pragma unroll 8
            for (int j = 0; j < D; ++j) {
                const float ki = K[i * Ds + j];
                kk = fmaf(K[t * Ds + j], ki, kk);
                qk = fmaf(Q[t * Ds + j], ki, qk);
            }
            const float ex = chunkmath::gate_exp(G[t] - G[i]);
            Af[t * kAs + i] = (i < t && t < n) ? Bt[t] * ex * kk : 0.f;
            P[t * kAs + i] = (i <= t && t < n) ? ex * qk : 0.f;
        }
        __syncthreads();
        chunkmath::solve_unit_lower<kThreads, kAs>(Af, X, tid, [] { __syncthreads(); });
        // W = T diag(beta e^G) K and Ut = T diag(beta) V
        for (int e = tid; e < kC * D; e += kThreads) {
            const int t = e / D, j = e % D;
            float w = 0.f, u = 0.f;
            for (int i = 0; i <= t; ++i) {
                const float tb = Af[t * kAs + i] * Bt[i];
                w = fmaf(tb * eG[i], K[i * Ds + j], w);
                u = fmaf(tb, V[i * Ds + j], u);
            }
            W[t * Ds + j] = w;
            U[t * Ds + j] = u;
        }
        __syncthreads();
        // U = Ut - W S^T
        for (int e = tid; e < kC * D; e += kThreads) {
            const int t = e / D, x = e % D;
            float acc = 0.f;
#pragma unroll 8
            for (int j = 0; j < D; ++j) acc = fmaf(W[t * Ds + j], S[x * Ds + j], acc);
            U[t * Ds + x] -= acc;
        }
        __syncthreads();
        // o = q_scale (e^{G_t} q_t S^T + sum_{i <= t} P[t][i] u_i), valid rows only
        for (int e = tid; e < n * D; e += kThreads) {
            const int t = e / D, x = e % D;
            float qs = 0.f, pu = 0.f;
#pragma unroll 8
            for (int j = 0; j < D; ++j) qs = fmaf(Q[t * Ds + j], S[x * Ds + j], qs);
            for (int i = 0; i <= t; ++i) pu = fmaf(P[t * kAs + i], U[i * Ds + x], pu);
            a.o[(size_t(t0 + t) * a.h_v + h) * D + x] = gdn::f32_to_bf16(a.q_scale * fmaf(eG[t], qs, pu));
        }
        // S' = e^{G_last} S + U^T diag(dec) K (new values held until every read of S is done)
        constexpr int kPer = (D * D + kThreads - 1) / kThreads;
        float nv[kPer];
        const float egl = eG[n - 1];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int e = tid + u * kThreads;
            if (e < D * D) {
                const int x = e / D, j = e % D;
                float acc = 0.f;
                for (int i = 0; i < n; ++i) acc = fmaf(U[i * Ds + x] * dec[i], K[i * Ds + j], acc);
                nv[u] = fmaf(egl, S[x * Ds + j], acc);
            }
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int e = tid + u * kThreads;
            if (e < D * D) S[(e / D) * Ds + e % D] = nv[u];
        }
        __syncthreads();
    }
    // Publication: only the final state, and not while the status word holds
    // GDN_DEV_TIMEOUT (results after a timed-out wait are not trusted).
    if (!a.status || !(*reinterpret_cast<volatile uint32_t *>(a.status) & GDN_DEV_TIMEOUT))
        for (int e = tid; e < D * D; e += kThreads)
            a.pool[size_t(dst) * a.slot_stride + head_off + e] = S[(e / D) * Ds + e % D];
}

template <int D>
int launch_small(const SmallArgs &a, long long grid, cudaStream_t st) {
    constexpr size_t smem = SmallLay<D>::kBytes;
    if (cudaFuncSetAttribute(gdn_prefill_small_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    gdn_prefill_small_kernel<D><<<unsigned(grid), kThreads, smem, st>>>(a);
    return gdn_host::launch_status(cudaGetLastError());
}

}  // namespace

// The fp32 chunk-form prefill for d in {16, 32, 64} (called by
// gdn_chunked_prefill after its argument checks and the length-order table).
int gdn_prefill_small_launch(const gdn_dims *dims, int32_t nseq, int32_t row_capacity, const int32_t *cu_seqlens,
                             const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v, const float *g,
                             const float *beta, float *pool_layer, int64_t slot_stride, int32_t num_slots,
                             const int32_t *src_slot, const int32_t *dst_slot, gdn_bf16 *o, const int32_t *order,
                             uint32_t *dev_status, cudaStream_t st) {
    SmallArgs a{};
    a.cu = cu_seqlens;
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
    a.order = order;
    a.q_scale = dims->q_scale;
    a.status = dev_status;
    const long long grid = (long long)nseq * dims->h_v;
    switch (dims->d_k) {
        case 16: return launch_small<16>(a, grid, st);
        case 32: return launch_small<32>(a, grid, st);
        case 64: return launch_small<64>(a, grid, st);
        default: return GDN_ERR_SHAPE;
    }
}
