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
    static constexpr int RB = kWarps * RPW;                  // state rows per CTA
    static constexpr size_t kTileOff = 128;
    static constexpr size_t kKqOff = kTileOff + size_t(RB) * DK * 4;
    static constexpr size_t kVOff = kKqOff + size_t(GDN_MAX_ROWS) * 2 * DK * 2;
    static constexpr size_t kGOff = kVOff + size_t(GDN_MAX_ROWS) * RB * 4;
    static constexpr size_t kSmem = kGOff + 2 * GDN_MAX_ROWS * 4;
    // replay mode (limited by instruction issue, not HBM): k and q staged as
    // fp32, converted once per CTA instead of once per lane group, and the
    // previous transaction's accepted rows (k as fp32, v, g, beta)
    static constexpr size_t kVOffR = kKqOff + size_t(GDN_MAX_ROWS) * 2 * DK * 4;
    static constexpr size_t kGOffR = kVOffR + size_t(GDN_MAX_ROWS) * RB * 4;
    static constexpr size_t kRkOff = kGOffR + 2 * GDN_MAX_ROWS * 4;
    static constexpr size_t kRvOff = kRkOff + size_t(GDN_MAX_ROWS) * DK * 4;
    static constexpr size_t kRgOff = kRvOff + size_t(GDN_MAX_ROWS) * RB * 4;
    static constexpr size_t kSmemReplay = kRgOff + 2 * GDN_MAX_ROWS * 4;
};

// Kernel modes: one token into a destination slot; K+1 rows with a
// checkpoint per row; the same reading the start state at an arena offset;
// replay of the previous transaction's accepted rows into the destination
// slot followed by outputs for the new rows.
enum { kDecode = 0, kVerify = 1, kVerifyAt = 2, kReplay = 3 };

struct RecArgs {
    const int32_t *cu_rows;
    const uint16_t *q, *k, *v;
    const float *g, *beta;
    const float *pool_src;
    float *pool_dst;
    int64_t slot_stride;
    int32_t num_slots;
    const int32_t *src_slot, *dst_slot;
    const int64_t *src_off;  // start state at pool_src + src_off[r] (located variant)
    int64_t max_off;         // largest valid src_off
    // replay mode: rows prev_cu[r] .. prev_cu[r] + prev_acc[r] of the previous transaction
    const int32_t *prev_cu, *prev_acc;
    const uint16_t *pk, *pv;
    const float *pg, *pbeta;
    int32_t prev_capacity;
    float *ckpt;
    uint64_t *ckpt_tag;
    uint32_t txn;
    uint16_t *o;
    uint32_t *status;
    int32_t B, h_qk, h_v, dv, row_capacity, grp, bph;
    float q_scale;
    // A later layer of a multi-layer call: the tables and this layer's state
    // tile are read before waiting for the previous layer's launch.  That is
    // safe because the previous layers write neither, and because the first
    // layer's launch (not early) does not let its successor start before
    // every earlier launch on the stream -- the commit that wrote the slots
    // -- has completed: a launch can only start once its predecessor has
    // started, so every later layer starts after that point too.
    int32_t early;
};

template <int LPR>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
}

// Packed pairs of fp32 (Blackwell's f32x2 arithmetic: two lanes of IEEE
// round-to-nearest fp32 per instruction, each rounded exactly like the
// scalar operation).
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// A lane's share of a row dot product: even and odd elements accumulate in
// the two halves of a packed pair (in element order), then the halves add.
template <int NV>
__device__ __forceinline__ float lane_dot(const float4 (&s)[NV], const float4 (&x)[NV]) {
    unsigned long long acc = f2_mul(f2_pack(s[0].x, s[0].y), f2_pack(x[0].x, x[0].y));
    acc = f2_fma(f2_pack(s[0].z, s[0].w), f2_pack(x[0].z, x[0].w), acc);
#pragma unroll
    for (int c = 1; c < NV; ++c) {
        acc = f2_fma(f2_pack(s[c].x, s[c].y), f2_pack(x[c].x, x[c].y), acc);
        acc = f2_fma(f2_pack(s[c].z, s[c].w), f2_pack(x[c].z, x[c].w), acc);
    }
    float e, o;
    f2_unpack(acc, e, o);
    return __fadd_rn(e, o);
}

// The state half of a token: prediction S k, then S <- alpha S + u k^T.
// row_update below performs exactly these operations and then the output dot
// product, so a replayed state is bit-identical to a verified checkpoint.
template <int NV, int LPR>
__device__ __forceinline__ void row_advance(float4 (&s)[NV], const float4 (&kf)[NV], float alpha, float b,
                                            float vv) {
    const float pred = group_sum<LPR>(lane_dot<NV>(s, kf));
    const float u = __fmul_rn(b, __fsub_rn(vv, __fmul_rn(alpha, pred)));
    // s <- u k + alpha s, elementwise (round(alpha s) then one fused multiply-add)
    const unsigned long long a2 = f2_pack(alpha, alpha), u2 = f2_pack(u, u);
#pragma unroll
    for (int c = 0; c < NV; ++c) {
        const unsigned long long xy =
            f2_fma(u2, f2_pack(kf[c].x, kf[c].y), f2_mul(a2, f2_pack(s[c].x, s[c].y)));
        const unsigned long long zw =
            f2_fma(u2, f2_pack(kf[c].z, kf[c].w), f2_mul(a2, f2_pack(s[c].z, s[c].w)));
        f2_unpack(xy, s[c].x, s[c].y);
        f2_unpack(zw, s[c].z, s[c].w);
    }
}

// One token for one state row held by a lane group.  Returns the row's
// output value (before q_scale).  Shared by decode and verify.
template <int NV, int LPR>
__device__ __forceinline__ float row_update(float4 (&s)[NV], const float4 (&kf)[NV], const float4 (&qf)[NV],
                                            float alpha, float b, float vv) {
    row_advance<NV, LPR>(s, kf, alpha, b, vv);
    return group_sum<LPR>(lane_dot<NV>(s, qf));
}

__device__ __forceinline__ float4 bf16x4_to_f32(uint2 w) {
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u), __uint_as_float(w.y << 16),
                       __uint_as_float(w.y & 0xffff0000u));
}

// Four CTAs per SM; replay (bound by its per-token chain rather than by HBM)
// is held to 48 registers so that five fit (its shared memory allows five).
template <int DK, int MODE>
__global__ void __launch_bounds__(kThreads, MODE == kReplay ? 5 : 4) gdn_recurrent_kernel(const RecArgs a) {
    using L = Lay<DK>;
    constexpr bool VERIFY = (MODE == kVerify || MODE == kVerifyAt);
    constexpr bool AT = (MODE == kVerifyAt);
    constexpr bool REPLAY = (MODE == kReplay);
    constexpr bool WRITES_SLOT = (MODE == kDecode || MODE == kReplay);
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    int *flag = reinterpret_cast<int *>(smem + 64);
    float *tile = reinterpret_cast<float *>(smem + L::kTileOff);
    uint16_t *kq = reinterpret_cast<uint16_t *>(smem + L::kKqOff);
    float *kqf = reinterpret_cast<float *>(smem + L::kKqOff);  // replay: fp32 k/q
    float *vsm = reinterpret_cast<float *>(smem + (REPLAY ? L::kVOffR : L::kVOff));
    float *gsm = reinterpret_cast<float *>(smem + (REPLAY ? L::kGOffR : L::kGOff));
    float *bsm = gsm + GDN_MAX_ROWS;
    // Programmatic dependent launch.  A first (non-early) launch waits for
    // everything before it on the stream (a commit writing the slots, say)
    // before it lets the next launch start; an early launch (a later layer of
    // a multi-layer call) lets the next layer start at once and waits only
    // once its own state tile's copy is under way (see RecArgs::early).
    if (a.early) {
        gdn::pdl_launch_dependents();
    } else {
        gdn::pdl_wait();
        gdn::pdl_launch_dependents();
    }

    const int tid = threadIdx.x;
    const int bid = blockIdx.x;
    const int rb = bid % a.bph;
    const int h = (bid / a.bph) % a.h_v;
    const int r = bid / (a.bph * a.h_v);
    const bool lead = (h == 0 && rb == 0 && tid == 0);

    // Every table entry this request needs, loaded together (no load waits
    // on another); then the checks.
    int t0 = r, t1 = r + 1;
    if (VERIFY || REPLAY) {
        t0 = a.cu_rows[r];
        t1 = a.cu_rows[r + 1];
    }
    int acc = -1, pc0 = 0, pc1 = 0;
    if (REPLAY) {
        acc = a.prev_acc[r];
        pc0 = a.prev_cu[r];
        pc1 = a.prev_cu[r + 1];
    }
    int64_t off = 0;
    int src = 0;
    if (AT)
        off = a.src_off[r];
    else
        src = a.src_slot[r];
    int dst = 0;
    if (WRITES_SLOT) dst = a.dst_slot[r];

    uint32_t bad = 0;
    const int nrows = t1 - t0;
    if (VERIFY || REPLAY) {
        const int min_rows = REPLAY ? 0 : 1;
        if (t0 < 0 || nrows < min_rows || nrows > GDN_MAX_ROWS || t1 > a.row_capacity) bad |= GDN_DEV_ROWS_BAD;
    }
    int p0 = 0, nrep = 0;  // replay rows p0 .. p0 + nrep - 1 of the previous transaction
    if (REPLAY && acc >= 0) {
        p0 = pc0;
        nrep = acc + 1;
        if (p0 < 0 || p0 + nrep > pc1 || nrep > GDN_MAX_ROWS || pc1 > a.prev_capacity) bad |= GDN_DEV_ROWS_BAD;
    }
    const float *src_base = a.pool_src;
    if (AT) {
        if (off < 0 || off > a.max_off || (off & 3) != 0)
            bad |= GDN_DEV_SLOT_OOR;
        else
            src_base = a.pool_src + off;
    } else {
        if (src < 0 || src >= a.num_slots)
            bad |= GDN_DEV_SLOT_OOR;
        else
            src_base = a.pool_src + size_t(src) * a.slot_stride;
    }
    if (WRITES_SLOT && (dst < 0 || dst >= a.num_slots)) bad |= GDN_DEV_SLOT_OOR;
    if (bad) {
        if (a.early) gdn::pdl_wait();
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
        gdn::bulk_g2s(tile, src_base + tile_off, uint32_t(nr) * DK * 4u, bar);
    }
    if (a.early) gdn::pdl_wait();  // the rows may come from the previous launch's outputs

    // Stage the rows: k and q (this request's qk-head, 16 B per load), the
    // tile's v entries and the gates, and in replay mode the previous
    // transaction's accepted k, v and gates.  Every thread issues all of its
    // loads before its first shared-memory store, so the loads overlap
    // instead of waiting on one another.
    const int hq = h / a.grp;
    constexpr int VPR = DK / 8;
    constexpr int KQ_IT = (GDN_MAX_ROWS * 2 * VPR + kThreads - 1) / kThreads;
    constexpr int V_IT = (GDN_MAX_ROWS * L::RB + kThreads - 1) / kThreads;
    constexpr int RK_IT = (GDN_MAX_ROWS * VPR + kThreads - 1) / kThreads;
    uint4 kqw[KQ_IT];
    float vw[V_IT];
#pragma unroll
    for (int j = 0; j < KQ_IT; ++j) {
        const int i = tid + j * kThreads;
        if (i < nrows * 2 * VPR) {
            const int t = i / (2 * VPR), rem = i % (2 * VPR), which = rem / VPR, c = rem % VPR;
            const uint16_t *sp = (which == 0 ? a.k : a.q) + (size_t(t0 + t) * a.h_qk + hq) * DK + c * 8;
            kqw[j] = __ldg(reinterpret_cast<const uint4 *>(sp));
        }
    }
#pragma unroll
    for (int j = 0; j < V_IT; ++j) {
        const int i = tid + j * kThreads;
        const int t = i / L::RB, row = i % L::RB;
        if (t < nrows && row < nr) vw[j] = gdn::bf16_to_f32(a.v[(size_t(t0 + t) * a.h_v + h) * a.dv + row0 + row]);
    }
    float gw = 0.f, bw = 0.f;
    if (tid < nrows) {
        gw = a.g[size_t(t0 + tid) * a.h_v + h];
        bw = a.beta[size_t(t0 + tid) * a.h_v + h];
    }
    float *rk = reinterpret_cast<float *>(smem + L::kRkOff);
    float *rv = reinterpret_cast<float *>(smem + L::kRvOff);
    float *rg = reinterpret_cast<float *>(smem + L::kRgOff);
    float *rbeta = rg + GDN_MAX_ROWS;
    uint4 rkw[RK_IT];
    float rvw[V_IT];
    float rgw = 0.f, rbw = 0.f;
    if constexpr (REPLAY) {
#pragma unroll
        for (int j = 0; j < RK_IT; ++j) {
            const int i = tid + j * kThreads;
            if (i < nrep * VPR) {
                const int t = i / VPR, c = i % VPR;
                rkw[j] = __ldg(reinterpret_cast<const uint4 *>(a.pk + (size_t(p0 + t) * a.h_qk + hq) * DK + c * 8));
            }
        }
#pragma unroll
        for (int j = 0; j < V_IT; ++j) {
            const int i = tid + j * kThreads;
            const int t = i / L::RB, row = i % L::RB;
            if (t < nrep && row < nr)
                rvw[j] = gdn::bf16_to_f32(a.pv[(size_t(p0 + t) * a.h_v + h) * a.dv + row0 + row]);
        }
        if (tid < nrep) {
            rgw = a.pg[size_t(p0 + tid) * a.h_v + h];
            rbw = a.pbeta[size_t(p0 + tid) * a.h_v + h];
        }
    }
    // ... then the stores.
#pragma unroll
    for (int j = 0; j < KQ_IT; ++j) {
        const int i = tid + j * kThreads;
        if (i < nrows * 2 * VPR) {
            const int t = i / (2 * VPR), rem = i % (2 * VPR), which = rem / VPR, c = rem % VPR;
            if constexpr (REPLAY) {
                float4 *dp = reinterpret_cast<float4 *>(kqf + (t * 2 + which) * DK + c * 8);
                dp[0] = bf16x4_to_f32(make_uint2(kqw[j].x, kqw[j].y));
                dp[1] = bf16x4_to_f32(make_uint2(kqw[j].z, kqw[j].w));
            } else {
                *reinterpret_cast<uint4 *>(kq + (t * 2 + which) * DK + c * 8) = kqw[j];
            }
        }
    }
#pragma unroll
    for (int j = 0; j < V_IT; ++j) {
        const int i = tid + j * kThreads;
        const int t = i / L::RB, row = i % L::RB;
        if (t < nrows && row < nr) vsm[t * L::RB + row] = vw[j];
    }
    if (tid < nrows) {
        gsm[tid] = expf(gw);  // alpha_t, once per token
        bsm[tid] = bw;
    }
    if constexpr (REPLAY) {
#pragma unroll
        for (int j = 0; j < RK_IT; ++j) {
            const int i = tid + j * kThreads;
            if (i < nrep * VPR) {
                const int t = i / VPR, c = i % VPR;
                float4 *dp = reinterpret_cast<float4 *>(rk + t * DK + c * 8);
                dp[0] = bf16x4_to_f32(make_uint2(rkw[j].x, rkw[j].y));
                dp[1] = bf16x4_to_f32(make_uint2(rkw[j].z, rkw[j].w));
            }
        }
#pragma unroll
        for (int j = 0; j < V_IT; ++j) {
            const int i = tid + j * kThreads;
            const int t = i / L::RB, row = i % L::RB;
            if (t < nrep && row < nr) rv[t * L::RB + row] = rvw[j];
        }
        if (tid < nrep) {
            rg[tid] = expf(rgw);
            rbeta[tid] = rbw;
        }
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
    const int lr = warp * L::RPW + gi;  // state row of this lane group within the tile
    const bool act = lr < nr;

    float4 s[L::NV];
#pragma unroll
    for (int c = 0; c < L::NV; ++c)
        s[c] = act ? *reinterpret_cast<const float4 *>(tile + lr * DK + (c * L::LPR + li) * 4)
                   : make_float4(0.f, 0.f, 0.f, 0.f);

    if (REPLAY) {
        // The previous transaction's accepted rows: the state half of each token.
        for (int t = 0; t < nrep; ++t) {
            const float alpha = rg[t];
            const float b = rbeta[t];
            float4 kf[L::NV];
#pragma unroll
            for (int c = 0; c < L::NV; ++c)
                kf[c] = *reinterpret_cast<const float4 *>(rk + t * DK + (c * L::LPR + li) * 4);
            const float vv = act ? rv[t * L::RB + lr] : 0.f;
            row_advance<L::NV, L::LPR>(s, kf, alpha, b, vv);
        }
        // The replayed state is the request's committed state (also copied
        // when nothing is pending but the request moves to a fresh slot).
        const bool moved = src != dst;
        if (act && (nrep > 0 || moved)) {
            float *dp = a.pool_dst + size_t(dst) * a.slot_stride + tile_off;
#pragma unroll
            for (int c = 0; c < L::NV; ++c) *reinterpret_cast<float4 *>(dp + lr * DK + (c * L::LPR + li) * 4) = s[c];
        }
    }
    for (int t = 0; t < nrows; ++t) {
        const float alpha = gsm[t];
        const float b = bsm[t];
        float4 kf[L::NV], qf[L::NV];
#pragma unroll
        for (int c = 0; c < L::NV; ++c) {
            if constexpr (REPLAY) {
                kf[c] = *reinterpret_cast<const float4 *>(kqf + (t * 2 + 0) * DK + (c * L::LPR + li) * 4);
                qf[c] = *reinterpret_cast<const float4 *>(kqf + (t * 2 + 1) * DK + (c * L::LPR + li) * 4);
            } else {
                kf[c] = bf16x4_to_f32(*reinterpret_cast<const uint2 *>(kq + (t * 2 + 0) * DK + (c * L::LPR + li) * 4));
                qf[c] = bf16x4_to_f32(*reinterpret_cast<const uint2 *>(kq + (t * 2 + 1) * DK + (c * L::LPR + li) * 4));
            }
        }
        const float vv = act ? vsm[t * L::RB + lr] : 0.f;
        const float e = row_update<L::NV, L::LPR>(s, kf, qf, alpha, b, vv);
        if (act) {
            const size_t orow = size_t(t0 + t) * a.h_v * a.dv + size_t(h) * a.dv + row0;
            if (li == 0) a.o[orow + lr] = gdn::f32_to_bf16(__fmul_rn(a.q_scale, e));
            if (VERIFY) {
                float *ck = a.ckpt + size_t(t0 + t) * state_elems + tile_off;
#pragma unroll
                for (int c = 0; c < L::NV; ++c)
                    __stcs(reinterpret_cast<float4 *>(ck + lr * DK + (c * L::LPR + li) * 4), s[c]);
            }
        }
    }
    if (MODE == kDecode && act) {
        float *dp = a.pool_dst + size_t(dst) * a.slot_stride + tile_off;
#pragma unroll
        for (int c = 0; c < L::NV; ++c) *reinterpret_cast<float4 *>(dp + lr * DK + (c * L::LPR + li) * 4) = s[c];
    }
    if (VERIFY && lead) a.ckpt_tag[r] = (uint64_t(a.txn) << 32) | uint32_t(nrows);
}

template <int DK, int MODE>
int launch(const RecArgs &a, cudaStream_t st) {
    using L = Lay<DK>;
    auto kern = gdn_recurrent_kernel<DK, MODE>;
    constexpr size_t smem = MODE == kReplay ? L::kSmemReplay : L::kSmem;
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
            return GDN_ERR_CUDA;
    }
    RecArgs b = a;
    b.bph = (a.dv + L::RB - 1) / L::RB;
    const long long grid = (long long)a.B * a.h_v * b.bph;
    if (grid <= 0) return GDN_OK;
    if (grid > 0x7fffffffLL) return GDN_ERR_ARG;
    return gdn_host::launch_pdl(kern, dim3(unsigned(grid)), dim3(kThreads), smem, st, b);
}

template <int MODE>
int dispatch(int dk, const RecArgs &a, cudaStream_t st) {
    switch (dk) {
        case 16: return launch<16, MODE>(a, st);
        case 32: return launch<32, MODE>(a, st);
        case 64: return launch<64, MODE>(a, st);
        case 128: return launch<128, MODE>(a, st);
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
    return dispatch<kDecode>(dims->d_k, a, static_cast<cudaStream_t>(stream));
}

static int gdn_verify_impl(int early, const gdn_dims *dims, int32_t B, int32_t row_capacity, const int32_t *cu_rows,
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
    a.early = early;
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
    return dispatch<kVerify>(dims->d_k, a, static_cast<cudaStream_t>(stream));
}

static int gdn_verify_at_impl(int early, const gdn_dims *dims, int32_t B, int32_t row_capacity, const int32_t *cu_rows,
                             const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v, const float *g,
                             const float *beta, const float *state_base, int64_t state_elems_total,
                             const int64_t *src_off, float *ckpt_layer, uint64_t *ckpt_tag, uint32_t txn, gdn_bf16 *o,
                             uint32_t *dev_status, void *stream) {
    if (!dims) return GDN_ERR_NULL;
    if (!gdn_host::dims_ok(dims)) return GDN_ERR_SHAPE;
    if (B < 0 || row_capacity < 0) return GDN_ERR_ARG;
    if (!q || !k || !v || !g || !beta || !state_base || !src_off || !cu_rows || !ckpt_layer || !ckpt_tag || !o)
        return GDN_ERR_NULL;
    const int64_t se = int64_t(dims->h_v) * dims->d_v * dims->d_k;
    if (state_elems_total < se) return GDN_ERR_ARG;
    if (!gdn_host::aligned16(q) || !gdn_host::aligned16(k) || !gdn_host::aligned16(state_base) ||
        !gdn_host::aligned16(ckpt_layer))
        return GDN_ERR_ARG;
    if (B == 0) return GDN_OK;
    RecArgs a{};
    a.early = early;
    a.cu_rows = cu_rows;
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.pool_src = state_base;
    a.src_off = src_off;
    a.max_off = state_elems_total - se;
    a.num_slots = 1;
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
    return dispatch<kVerifyAt>(dims->d_k, a, static_cast<cudaStream_t>(stream));
}

static int gdn_verify_replay_impl(int early, const gdn_dims *dims, int32_t B, int32_t row_capacity, const int32_t *cu_rows,
                                 const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v, const float *g,
                                 const float *beta, int32_t prev_capacity, const int32_t *prev_cu_rows,
                                 const int32_t *prev_accept_len, const gdn_bf16 *prev_k, const gdn_bf16 *prev_v,
                                 const float *prev_g, const float *prev_beta, float *pool_layer, int64_t slot_stride,
                                 int32_t num_slots, const int32_t *src_slot, const int32_t *dst_slot, gdn_bf16 *o,
                                 uint32_t *dev_status, void *stream) {
    int st = common_checks(dims, B, q, k, v, g, beta, pool_layer, slot_stride, num_slots, src_slot, o);
    if (st != GDN_OK) return st;
    if (!cu_rows || !dst_slot || !prev_cu_rows || !prev_accept_len || !prev_k || !prev_v || !prev_g || !prev_beta)
        return GDN_ERR_NULL;
    if (row_capacity < 0 || prev_capacity < 0) return GDN_ERR_ARG;
    if (!gdn_host::aligned16(prev_k)) return GDN_ERR_ARG;
    if (B == 0) return GDN_OK;
    RecArgs a{};
    a.early = early;
    a.cu_rows = cu_rows;
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
    a.prev_cu = prev_cu_rows;
    a.prev_acc = prev_accept_len;
    a.pk = prev_k;
    a.pv = prev_v;
    a.pg = prev_g;
    a.pbeta = prev_beta;
    a.prev_capacity = prev_capacity;
    a.o = o;
    a.status = dev_status;
    a.B = B;
    a.h_qk = dims->h_qk;
    a.h_v = dims->h_v;
    a.dv = dims->d_v;
    a.row_capacity = row_capacity;
    a.grp = dims->h_v / dims->h_qk;
    a.q_scale = dims->q_scale;
    return dispatch<kReplay>(dims->d_k, a, static_cast<cudaStream_t>(stream));
}

extern "C" int gdn_verify(const gdn_dims *dims, int32_t B, int32_t row_capacity, const int32_t *cu_rows,
                          const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v, const float *g,
                          const float *beta, const float *pool_layer, int64_t slot_stride, int32_t num_slots,
                          const int32_t *src_slot, float *ckpt_layer, uint64_t *ckpt_tag, uint32_t txn,
                          gdn_bf16 *o, uint32_t *dev_status, void *stream) {
    return gdn_verify_impl(0, dims, B, row_capacity, cu_rows, q, k, v, g, beta, pool_layer, slot_stride, num_slots, src_slot, ckpt_layer, ckpt_tag, txn, o, dev_status, stream);
}

extern "C" int gdn_verify_at(const gdn_dims *dims, int32_t B, int32_t row_capacity, const int32_t *cu_rows,
                             const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v, const float *g,
                             const float *beta, const float *state_base, int64_t state_elems_total,
                             const int64_t *src_off, float *ckpt_layer, uint64_t *ckpt_tag, uint32_t txn, gdn_bf16 *o,
                             uint32_t *dev_status, void *stream) {
    return gdn_verify_at_impl(0, dims, B, row_capacity, cu_rows, q, k, v, g, beta, state_base, state_elems_total, src_off, ckpt_layer, ckpt_tag, txn, o, dev_status, stream);
}

extern "C" int gdn_verify_replay(const gdn_dims *dims, int32_t B, int32_t row_capacity, const int32_t *cu_rows,
                                 const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v, const float *g,
                                 const float *beta, int32_t prev_capacity, const int32_t *prev_cu_rows,
                                 const int32_t *prev_accept_len, const gdn_bf16 *prev_k, const gdn_bf16 *prev_v,
                                 const float *prev_g, const float *prev_beta, float *pool_layer, int64_t slot_stride,
                                 int32_t num_slots, const int32_t *src_slot, const int32_t *dst_slot, gdn_bf16 *o,
                                 uint32_t *dev_status, void *stream) {
    return gdn_verify_replay_impl(0, dims, B, row_capacity, cu_rows, q, k, v, g, beta, prev_capacity, prev_cu_rows, prev_accept_len, prev_k, prev_v, prev_g, prev_beta, pool_layer, slot_stride, num_slots, src_slot, dst_slot, o, dev_status, stream);
}

// Multi-layer issue of the per-layer verify calls: one host call walks the
// layers in order and makes the same calls a caller would make layer by
// layer (same kernels, arguments and stream).  A layer after the first may
// read its tables and start its state tile's copy before the previous
// layer's launch has finished (the rows still wait for it): the layers
// write none of them, and the first layer lets no successor start until
// every launch queued before the call (a commit, a prefill) is complete.
extern "C" int gdn_verify_layers(const gdn_dims *dims, int32_t num_layers, int32_t B, int32_t row_capacity,
                                 const int32_t *cu_rows, const gdn_layer_rows *rows, const float *pool,
                                 int64_t slot_stride, int64_t layer_stride, int32_t num_slots,
                                 const int32_t *src_slot, float *ckpt, int64_t ckpt_layer_stride,
                                 uint64_t *ckpt_tag, uint32_t txn, gdn_bf16 *o, int64_t o_layer_stride,
                                 uint32_t *dev_status, void *stream) {
    if (num_layers < 0) return GDN_ERR_ARG;
    if (num_layers > 0 && (!rows || !pool || !ckpt || !ckpt_tag || !o)) return GDN_ERR_NULL;
    for (int32_t l = 0; l < num_layers; ++l) {
        const gdn_layer_rows &x = rows[l];
        const int st = gdn_verify_impl(l > 0, dims, B, row_capacity, cu_rows, x.q, x.k, x.v, x.g, x.beta,
                                  pool + int64_t(l) * layer_stride, slot_stride, num_slots, src_slot,
                                  ckpt + int64_t(l) * ckpt_layer_stride, ckpt_tag + int64_t(l) * B, txn,
                                  o + int64_t(l) * o_layer_stride, dev_status, stream);
        if (st != GDN_OK) return st;
    }
    return GDN_OK;
}

extern "C" int gdn_verify_replay_layers(const gdn_dims *dims, int32_t num_layers, int32_t B, int32_t row_capacity,
                                        const int32_t *cu_rows, const gdn_layer_rows *rows, int32_t prev_capacity,
                                        const int32_t *prev_cu_rows, const int32_t *prev_accept_len,
                                        const gdn_layer_rows *prev_rows, float *pool, int64_t slot_stride,
                                        int64_t layer_stride, int32_t num_slots, const int32_t *src_slot,
                                        const int32_t *dst_slot, gdn_bf16 *o, int64_t o_layer_stride,
                                        uint32_t *dev_status, void *stream) {
    if (num_layers < 0) return GDN_ERR_ARG;
    if (num_layers > 0 && (!rows || !prev_rows || !pool || !o)) return GDN_ERR_NULL;
    for (int32_t l = 0; l < num_layers; ++l) {
        const gdn_layer_rows &x = rows[l];
        const gdn_layer_rows &p = prev_rows[l];
        const int st = gdn_verify_replay_impl(l > 0, dims, B, row_capacity, cu_rows, x.q, x.k, x.v, x.g, x.beta, prev_capacity,
                                         prev_cu_rows, prev_accept_len, p.k, p.v, p.g, p.beta,
                                         pool + int64_t(l) * layer_stride, slot_stride, num_slots, src_slot, dst_slot,
                                         o + int64_t(l) * o_layer_stride, dev_status, stream);
        if (st != GDN_OK) return st;
    }
    return GDN_OK;
}

extern "C" int gdn_verify_at_layers(const gdn_dims *dims, int32_t num_layers, int32_t B, int32_t row_capacity,
                                    const int32_t *cu_rows, const gdn_layer_rows *rows, const float *state_base,
                                    int64_t state_elems_total, const int64_t *src_off, float *ckpt,
                                    int64_t ckpt_layer_stride, uint64_t *ckpt_tag, uint32_t txn, gdn_bf16 *o,
                                    int64_t o_layer_stride, uint32_t *dev_status, void *stream) {
    if (num_layers < 0) return GDN_ERR_ARG;
    if (num_layers > 0 && (!rows || !src_off || !ckpt || !ckpt_tag || !o)) return GDN_ERR_NULL;
    for (int32_t l = 0; l < num_layers; ++l) {
        const gdn_layer_rows &x = rows[l];
        const int st = gdn_verify_at_impl(l > 0, dims, B, row_capacity, cu_rows, x.q, x.k, x.v, x.g, x.beta, state_base,
                                     state_elems_total, src_off + int64_t(l) * B,
                                     ckpt + int64_t(l) * ckpt_layer_stride, ckpt_tag + int64_t(l) * B, txn,
                                     o + int64_t(l) * o_layer_stride, dev_status, stream);
        if (st != GDN_OK) return st;
    }
    return GDN_OK;
}
