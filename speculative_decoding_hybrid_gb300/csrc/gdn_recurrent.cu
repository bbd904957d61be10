// Gated delta-rule decode step and fused K-draft verification (sm_103a).
//
// Operation ("Native three-step MTP", What changed: GDN state update with FP32
// gates, identical rounding in decode and verification; "Run chained MTP
// drafting in the batch Engine", Correctness fix: per-row recurrent
// checkpoints that let a rejected draft be rolled back):
//     S_t = alpha_t S_{t-1} + u_t k_t^T,  u_t = beta_t (v_t - alpha_t S_{t-1} k_t)
//     o_t = q_scale * S_t q_t,            alpha_t = expf(g_t)
// which is S_{t-1} alpha (I - beta k k^T) + beta v k^T written row by row:
// row a of S only needs k_t, q_t and the scalar v_t[a].
//
// Work decomposition: one CTA per (request, v-head, tile of RB state rows).
// The tile (RB x d_k fp32, contiguous in the slot) is brought into shared
// memory by one bulk asynchronous copy (TMA engine) while the threads stage
// the request's k/q rows (bf16), the tile's v entries and the gates.  Each
// state row then lives in the registers of LPR lanes (float4 slices, 128 B
// contiguous per lane group, so every global access is coalesced); the two
// dot products per token (S k before the update, S q after it) are lane-local
// FMAs plus an xor-shuffle tree over the group.  Verify streams the state
// after every row to its checkpoint; decode writes the final state to the
// destination slot.  Both run the same inline update with explicit
// round-to-nearest intrinsics, so verify's checkpoint j is bit-identical to
// j+1 decode steps.
//
// HBM roofline: per (request, layer) verify reads S_bytes and writes
// rows*S_bytes (+ ~24.8 KB of row I/O per row at 32 heads x 128); ~1.2 FP32
// flop per byte, far below the FP32 ridge, so the kernel is bandwidth-bound.
#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int DK>
struct Lay {
    static constexpr int LPR = (DK / 4) < 8 ? (DK / 4) : 8;  // lanes per state row
    static constexpr int NV = DK / (4 * LPR);                // float4 slices per lane
    static constexpr int RPW = 32 / LPR;                     // rows per warp per pass
    static constexpr int RPP = kWarps * RPW;                 // rows per CTA pass
    static constexpr int PASSES = 2;
    static constexpr int RB = RPP * PASSES;                  // state rows per CTA
    static constexpr size_t kTileOff = 128;
    static constexpr size_t kKqOff = kTileOff + size_t(RB) * DK * 4;
    static constexpr size_t kVOff = kKqOff + size_t(GDN_MAX_ROWS) * 2 * DK * 2;
    static constexpr size_t kGOff = kVOff + size_t(GDN_MAX_ROWS) * RB * 4;
    static constexpr size_t kSmem = kGOff + 2 * GDN_MAX_ROWS * 4;
};

struct RecArgs {
    const int32_t *cu_rows;
    const uint16_t *q, *k, *v;
    const float *g, *beta;
    const float *pool_src;
    float *pool_dst;
    int64_t slot_stride;
    int32_t num_slots;
    const int32_t *src_slot, *dst_slot;
    float *ckpt;
    uint64_t *ckpt_tag;
    uint32_t txn;
    uint16_t *o;
    uint32_t *status;
    int32_t B, h_qk, h_v, dv, row_capacity, grp, bph;
    float q_scale;
};

template <int LPR>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
}

template <int NV>
__device__ __forceinline__ float lane_dot(const float4 (&s)[NV], const float4 (&x)[NV]) {
    float acc = __fmul_rn(s[0].x, x[0].x);
    acc = __fmaf_rn(s[0].y, x[0].y, acc);
    acc = __fmaf_rn(s[0].z, x[0].z, acc);
    acc = __fmaf_rn(s[0].w, x[0].w, acc);
#pragma unroll
    for (int c = 1; c < NV; ++c) {
        acc = __fmaf_rn(s[c].x, x[c].x, acc);
        acc = __fmaf_rn(s[c].y, x[c].y, acc);
        acc = __fmaf_rn(s[c].z, x[c].z, acc);
        acc = __fmaf_rn(s[c].w, x[c].w, acc);
    }
    return acc;
}

// One token for one state row held by a lane group.  Returns the row's
// output value (before q_scale).  Shared by decode and verify.
template <int NV, int LPR>
__device__ __forceinline__ float row_update(float4 (&s)[NV], const float4 (&kf)[NV], const float4 (&qf)[NV],
                                            float alpha, float b, float vv) {
    const float pred = group_sum<LPR>(lane_dot<NV>(s, kf));
    const float u = __fmul_rn(b, __fsub_rn(vv, __fmul_rn(alpha, pred)));
#pragma unroll
    for (int c = 0; c < NV; ++c) {
        s[c].x = __fmaf_rn(u, kf[c].x, __fmul_rn(alpha, s[c].x));
        s[c].y = __fmaf_rn(u, kf[c].y, __fmul_rn(alpha, s[c].y));
        s[c].z = __fmaf_rn(u, kf[c].z, __fmul_rn(alpha, s[c].z));
        s[c].w = __fmaf_rn(u, kf[c].w, __fmul_rn(alpha, s[c].w));
    }
    return group_sum<LPR>(lane_dot<NV>(s, qf));
}

__device__ __forceinline__ float4 bf16x4_to_f32(uint2 w) {
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u), __uint_as_float(w.y << 16),
                       __uint_as_float(w.y & 0xffff0000u));
}

template <int DK, bool VERIFY>
__global__ void __launch_bounds__(kThreads, 2) gdn_recurrent_kernel(const RecArgs a) {
    using L = Lay<DK>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    int *flag = reinterpret_cast<int *>(smem + 64);
    float *tile = reinterpret_cast<float *>(smem + L::kTileOff);
    uint16_t *kq = reinterpret_cast<uint16_t *>(smem + L::kKqOff);
    float *vsm = reinterpret_cast<float *>(smem + L::kVOff);
    float *gsm = reinterpret_cast<float *>(smem + L::kGOff);
    float *bsm = gsm + GDN_MAX_ROWS;

    const int tid = threadIdx.x;
    const int bid = blockIdx.x;
    const int rb = bid % a.bph;
    const int h = (bid / a.bph) % a.h_v;
    const int r = bid / (a.bph * a.h_v);
    const bool lead = (h == 0 && rb == 0 && tid == 0);

    int t0, nrows;
    uint32_t bad = 0;
    if (VERIFY) {
        t0 = a.cu_rows[r];
        const int t1 = a.cu_rows[r + 1];
        nrows = t1 - t0;
        if (t0 < 0 || nrows < 1 || nrows > GDN_MAX_ROWS || t1 > a.row_capacity) bad |= GDN_DEV_ROWS_BAD;
    } else {
        t0 = r;
        nrows = 1;
    }
    const int src = a.src_slot[r];
    if (src < 0 || src >= a.num_slots) bad |= GDN_DEV_SLOT_OOR;
    int dst = 0;
    if (!VERIFY) {
        dst = a.dst_slot[r];
        if (dst < 0 || dst >= a.num_slots) bad |= GDN_DEV_SLOT_OOR;
    }
    if (bad) {
        if (lead) {
            gdn::set_status(a.status, bad);
            if (VERIFY) a.ckpt_tag[r] = uint64_t(a.txn) << 32;
        }
        return;
    }

    const int row0 = rb * L::RB;
    const int nr = min(L::RB, a.dv - row0);
    const size_t state_elems = size_t(a.h_v) * a.dv * DK;
    const size_t tile_off = size_t(h) * a.dv * DK + size_t(row0) * DK;

    if (tid == 0) {
        gdn::mbar_init(bar, 1);
        gdn::mbar_arrive_expect_tx(bar, uint32_t(nr) * DK * 4u);
        gdn::bulk_g2s(tile, a.pool_src + size_t(src) * a.slot_stride + tile_off, uint32_t(nr) * DK * 4u, bar);
    }

    // Stage k and q rows (bf16) of this request's qk-head, 16 B per load.
    const int hq = h / a.grp;
    constexpr int VPR = DK / 8;
    for (int i = tid; i < nrows * 2 * VPR; i += kThreads) {
        const int t = i / (2 * VPR);
        const int rem = i - t * 2 * VPR;
        const int which = rem / VPR;
        const int c = rem - which * VPR;
        const uint16_t *sp = (which == 0 ? a.k : a.q) + (size_t(t0 + t) * a.h_qk + hq) * DK + c * 8;
        *reinterpret_cast<uint4 *>(kq + (t * 2 + which) * DK + c * 8) = __ldg(reinterpret_cast<const uint4 *>(sp));
    }
    for (int i = tid; i < nrows * nr; i += kThreads) {
        const int t = i / nr;
        const int row = i - t * nr;
        vsm[t * L::RB + row] = gdn::bf16_to_f32(a.v[(size_t(t0 + t) * a.h_v + h) * a.dv + row0 + row]);
    }
    if (tid < nrows) {
        gsm[tid] = a.g[size_t(t0 + tid) * a.h_v + h];
        bsm[tid] = a.beta[size_t(t0 + tid) * a.h_v + h];
    }
    if (tid == 0) *flag = gdn::mbar_wait_bounded(bar, 0) ? 1 : 0;
    __syncthreads();
    if (*flag == 0) {
        if (tid == 0) gdn::set_status(a.status, GDN_DEV_TIMEOUT);
        return;
    }
    (void)gdn::mbar_try_wait(bar, 0);  // phase already complete: acquire for this thread

    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int gi = lane / L::LPR;
    const int li = lane - gi * L::LPR;

    float4 s[L::PASSES][L::NV];
    int lr[L::PASSES];
    bool act[L::PASSES];
#pragma unroll
    for (int p = 0; p < L::PASSES; ++p) {
        lr[p] = p * L::RPP + warp * L::RPW + gi;
        act[p] = lr[p] < nr;
#pragma unroll
        for (int c = 0; c < L::NV; ++c)
            s[p][c] = act[p] ? *reinterpret_cast<const float4 *>(tile + lr[p] * DK + (c * L::LPR + li) * 4)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    for (int t = 0; t < nrows; ++t) {
        const float alpha = expf(gsm[t]);
        const float b = bsm[t];
        float4 kf[L::NV], qf[L::NV];
#pragma unroll
        for (int c = 0; c < L::NV; ++c) {
            kf[c] = bf16x4_to_f32(*reinterpret_cast<const uint2 *>(kq + (t * 2 + 0) * DK + (c * L::LPR + li) * 4));
            qf[c] = bf16x4_to_f32(*reinterpret_cast<const uint2 *>(kq + (t * 2 + 1) * DK + (c * L::LPR + li) * 4));
        }
        const size_t orow = size_t(t0 + t) * a.h_v * a.dv + size_t(h) * a.dv + row0;
        float *ck = VERIFY ? a.ckpt + size_t(t0 + t) * state_elems + tile_off : nullptr;
#pragma unroll
        for (int p = 0; p < L::PASSES; ++p) {
            const float vv = act[p] ? vsm[t * L::RB + lr[p]] : 0.f;
            const float e = row_update<L::NV, L::LPR>(s[p], kf, qf, alpha, b, vv);
            if (act[p]) {
                if (li == 0) a.o[orow + lr[p]] = gdn::f32_to_bf16(__fmul_rn(a.q_scale, e));
                if (VERIFY) {
#pragma unroll
                    for (int c = 0; c < L::NV; ++c)
                        __stcs(reinterpret_cast<float4 *>(ck + lr[p] * DK + (c * L::LPR + li) * 4), s[p][c]);
                }
            }
        }
    }
    if (!VERIFY) {
        float *dp = a.pool_dst + size_t(dst) * a.slot_stride + tile_off;
#pragma unroll
        for (int p = 0; p < L::PASSES; ++p)
            if (act[p]) {
#pragma unroll
                for (int c = 0; c < L::NV; ++c)
                    *reinterpret_cast<float4 *>(dp + lr[p] * DK + (c * L::LPR + li) * 4) = s[p][c];
            }
    }
    if (VERIFY && lead) a.ckpt_tag[r] = (uint64_t(a.txn) << 32) | uint32_t(nrows);
}

template <int DK, bool VERIFY>
int launch(const RecArgs &a, cudaStream_t st) {
    using L = Lay<DK>;
    auto kern = gdn_recurrent_kernel<DK, VERIFY>;
    if (L::kSmem > 48 * 1024) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(L::kSmem)) != cudaSuccess)
            return GDN_ERR_CUDA;
    }
    RecArgs b = a;
    b.bph = (a.dv + L::RB - 1) / L::RB;
    const long long grid = (long long)a.B * a.h_v * b.bph;
    if (grid <= 0) return GDN_OK;
    if (grid > 0x7fffffffLL) return GDN_ERR_ARG;
    kern<<<unsigned(grid), kThreads, L::kSmem, st>>>(b);
    return gdn_host::launch_status(cudaGetLastError());
}

template <bool VERIFY>
int dispatch(int dk, const RecArgs &a, cudaStream_t st) {
    switch (dk) {
        case 16: return launch<16, VERIFY>(a, st);
        case 32: return launch<32, VERIFY>(a, st);
        case 64: return launch<64, VERIFY>(a, st);
        case 128: return launch<128, VERIFY>(a, st);
        default: return GDN_ERR_SHAPE;
    }
}

int common_checks(const gdn_dims *dims, int32_t B, const void *q, const void *k, const void *v, const void *g,
                  const void *beta, const void *pool, int64_t slot_stride, int32_t num_slots, const void *src,
                  const void *o) {
    if (!dims) return GDN_ERR_NULL;
    if (!gdn_host::dims_ok(dims)) return GDN_ERR_SHAPE;
    if (B < 0 || num_slots <= 0) return GDN_ERR_ARG;
    if (!q || !k || !v || !g || !beta || !pool || !src || !o) return GDN_ERR_NULL;
    const int64_t se = int64_t(dims->h_v) * dims->d_v * dims->d_k;
    if (slot_stride < se || (slot_stride % 4) != 0) return GDN_ERR_ARG;
    if (!gdn_host::aligned16(q) || !gdn_host::aligned16(k) || !gdn_host::aligned16(pool)) return GDN_ERR_ARG;
    return GDN_OK;
}

}  // namespace

extern "C" int gdn_decode_step(const gdn_dims *dims, int32_t B, const gdn_bf16 *q, const gdn_bf16 *k,
                               const gdn_bf16 *v, const float *g, const float *beta, float *pool_layer,
                               int64_t slot_stride, int32_t num_slots, const int32_t *src_slot,
                               const int32_t *dst_slot, gdn_bf16 *o, uint32_t *dev_status, void *stream) {
    int st = common_checks(dims, B, q, k, v, g, beta, pool_layer, slot_stride, num_slots, src_slot, o);
    if (st != GDN_OK) return st;
    if (!dst_slot) return GDN_ERR_NULL;
    if (B == 0) return GDN_OK;
    RecArgs a{};
    a.cu_rows = nullptr;
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.pool_src = pool_layer;
    a.pool_dst = pool_layer;
    a.slot_stride = slot_stride;
    a.num_slots = num_slots;
    a.src_slot = src_slot;
    a.dst_slot = dst_slot;
    a.o = o;
    a.status = dev_status;
    a.B = B;
    a.h_qk = dims->h_qk;
    a.h_v = dims->h_v;
    a.dv = dims->d_v;
    a.row_capacity = B;
    a.grp = dims->h_v / dims->h_qk;
    a.q_scale = dims->q_scale;
    return dispatch<false>(dims->d_k, a, static_cast<cudaStream_t>(stream));
}

extern "C" int gdn_verify(const gdn_dims *dims, int32_t B, int32_t row_capacity, const int32_t *cu_rows,
                          const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v, const float *g,
                          const float *beta, const float *pool_layer, int64_t slot_stride, int32_t num_slots,
                          const int32_t *src_slot, float *ckpt_layer, uint64_t *ckpt_tag, uint32_t txn,
                          gdn_bf16 *o, uint32_t *dev_status, void *stream) {
    int st = common_checks(dims, B, q, k, v, g, beta, pool_layer, slot_stride, num_slots, src_slot, o);
    if (st != GDN_OK) return st;
    if (!cu_rows || !ckpt_layer || !ckpt_tag) return GDN_ERR_NULL;
    if (row_capacity < 0) return GDN_ERR_ARG;
    if (!gdn_host::aligned16(ckpt_layer)) return GDN_ERR_ARG;
    if (B == 0) return GDN_OK;
    RecArgs a{};
    a.cu_rows = cu_rows;
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.pool_src = pool_layer;
    a.pool_dst = nullptr;
    a.slot_stride = slot_stride;
    a.num_slots = num_slots;
    a.src_slot = src_slot;
    a.ckpt = ckpt_layer;
    a.ckpt_tag = ckpt_tag;
    a.txn = txn;
    a.o = o;
    a.status = dev_status;
    a.B = B;
    a.h_qk = dims->h_qk;
    a.h_v = dims->h_v;
    a.dv = dims->d_v;
    a.row_capacity = row_capacity;
    a.grp = dims->h_v / dims->h_qk;
    a.q_scale = dims->q_scale;
    return dispatch<true>(dims->d_k, a, static_cast<cudaStream_t>(stream));
}
