// Chunked (WY/UT) GatedDeltaNet prefill (sm_103a): one fused kernel.
//
// "Run chained MTP drafting in the batch Engine", Correctness fix: the
// chunked plan runs a whole prompt at once and publishes only its final
// state (no per-row checkpoints).  Within a chunk of C = 64 tokens with start
// state S (d_v x d_k) and G = cumsum(g) (the chunk form of the gated delta
// rule):
//   A[t][i] = beta_t e^{G_t-G_i} k_t.k_i  (i < t),   T = (I + A)^{-1}
//   W  = T diag(beta e^G) K,   Ut = T diag(beta) V,   U = Ut - W S^T
//   O  = diag(e^G) Q S^T + (M o Q K^T) U,   M[t][i] = e^{G_t-G_i} (i <= t)
//   S' = e^{G_last} S + U^T diag(dec) K,    dec_i = e^{G_last-G_i}
//
// One CTA (16 warps) per (sequence, v-head) walks the sequence's chunks; the
// state stays on chip from the first chunk to the last, and no intermediate
// quantity leaves the SM (no workspace round trip through HBM).  All products
// run on the 5th-generation tensor cores (tcgen05, kind::f16, fp32
// accumulators in tensor memory).  Iteration c overlaps the state-dependent
// work of chunk c (the "scan": U, O, S') with the state-independent work of
// chunk c+1 (the "producer": [K;Q] K^T, A and P, T, W and Ut), in four slots:
//   1  MMA  phase A(c): U^T += -S W^T;  MMA1(c+1): [K;Q] K^T
//      SIMT the outputs of chunk c-1, o = e^G Oi + Oa (while phase A runs)
//   2  SIMT U^T -> bf16 parts of U and of U diag(dec) (tensor memory);
//           A(c+1) (fp32, shared) and P(c+1) (bf16 parts)
//   3  MMA  phase B(c): Oa = U^T P^T, dS = (U^T diag(dec)) K  (A from tensor
//           memory), then Oi(c) = S Q^T
//      SIMT T(c+1) = (I + A)^{-1}, then the operands T diag(beta e^G), T diag(beta)
//   4  MMA  MMA2(c+1): W^T = K^T (T diag(beta e^G))^T,  Ut^T = V^T (T diag(beta))^T
//      SIMT S <- e^{G_last} S + dS (fp32 in registers, bf16 parts in shared);
//           W^T(c+1) -> bf16 parts;  tensor copies of chunk c+2's K, Q and V
// Operands that are not exact bf16 (S, U, W, P, T-derived tiles) are split
// into two bf16 parts x = x1 + x2 and every product keeps the terms
// a1 b1 + a1 b2 + a2 b1 (or a1 b + a2 b when b is exact: q, k, v).
#include <cuda.h>

#include "common.cuh"
#include "chunk_math.cuh"
#include "tc.cuh"

namespace {

constexpr int kC = 64;              // chunk length
constexpr int kD = 128;             // d_k = d_v of this kernel
constexpr int kSimt = 512;          // warps 0..15: 4 per tensor-memory lane quadrant
constexpr int kThreads = kSimt + 32;  // + warp 16, which issues the copies and the products
constexpr int kCtl = kSimt / 32;
constexpr int kAs = 68;             // row stride (floats) of the fp32 matrix A -> T

// Barrier 1 over the 16 SIMT warps only (barrier 0 is the whole CTA's).
__device__ __forceinline__ void simt_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }

struct PrefArgs {
    const int32_t *cu;
    int32_t nseq, h_qk, h_v, grp, row_capacity, num_slots;
    const float *g, *beta;
    float *pool;
    int64_t slot_stride;
    const int32_t *src_slot, *dst_slot;
    uint16_t *o;
    const int32_t *order;  // sequences by decreasing length (gdn_prefill_order_kernel)
    float q_scale;
    uint32_t *status;
    uint64_t wait_ns;      // bound of every wait on a copy or a product
    int32_t withhold;      // self-test only: the last chunk's K/Q copy is never issued
    // q, k (rows x h_qk x 128) and v (rows x h_v x 128) as 3-D bf16 tensors
    // for the copy engine: boxes of 64 columns x 1 head x 64 rows, 128-byte
    // swizzle (the operand-tile layout), zero fill past row_capacity
    CUtensorMap tm_q, tm_k, tm_v;
};

// Shared-memory map (bytes from a 1024-aligned base).  Operand tiles are
// 128-byte-swizzled bf16 tiles (tc.cuh); K-major unless marked MN-major.
namespace smap {
constexpr uint32_t kS1 = 0, kS2 = 32768;   // S parts: 128 rows (d_v) x 128 (d_k), two 64-column atoms
// [K;Q] of a chunk, one per chunk parity: atom a (16 KB) holds K rows 0..63
// then Q rows 0..63 of columns 64a..64a+63.  Read as: the M = 128 A operand
// [K;Q] and the N = 64 B operand K (MMA1), MN-major K^T (MMA2) and K (phase
// B), and Q as the N = 64 B operand (phase A).
constexpr uint32_t kKQ = 65536;
constexpr uint32_t kV = 131072;            // V: 64 rows x 128, atoms 8 KB apart; MN-major V^T in MMA2
constexpr uint32_t kP = 147456;            // P parts (P1 then P2, 64 rows t x 64 i), one pair per parity
constexpr uint32_t kX = 180224;            // 32 KB, shared in turn by:
constexpr uint32_t kScratch = kX + 64 * kAs * 4;  //   A -> T (fp32 [64][kAs]) and a 4.5 KB scratch,
constexpr uint32_t kBW1 = kX, kBW2 = kX + 8192;   //   T diag(beta e^G) parts (64 rows t x 64 i),
constexpr uint32_t kBU1 = kX + 16384, kBU2 = kX + 24576;  // T diag(beta) parts,
constexpr uint32_t kW1 = kX, kW2 = kX + 16384;    //   W parts, MN-major: 128 rows d x 64 t
constexpr uint32_t kMisc = 212992;
// per chunk parity b (64 fp32 each, +256 b): G, e^G, dec, raw g, raw beta
constexpr uint32_t kG = kMisc, kEG = kMisc + 512, kDec = kMisc + 1024, kGraw = kMisc + 1536,
                   kBraw = kMisc + 2048;
constexpr uint32_t kBars = kMisc + 2560;   // mbarriers (16 slots)
constexpr uint32_t kTbase = kMisc + 2688;
constexpr uint32_t kFlags = kMisc + 2704;  // four rotating wait-result flags
constexpr uint32_t kAbort = kMisc + 2720;  // set by any thread whose bounded wait ran out
constexpr size_t kSmem = size_t(kMisc) + 2752 + 1024;  // + alignment slack
}  // namespace smap

// Tensor-memory columns (512): fp32 accumulators, then packed bf16 A operands.
namespace tcol {
constexpr uint32_t kU = 0;      // U^T (lanes d_v, columns t): Ut^T from MMA2, then += -S W^T
constexpr uint32_t kOi = 64;    // S Q^T
constexpr uint32_t kOa = 128;   // U^T P^T
constexpr uint32_t kdS = 192;   // (U^T diag(dec)) K, 128 columns
constexpr uint32_t kD1 = 320;   // [K;Q] K^T (lanes t, then q rows), later W^T (lanes d_k)
constexpr uint32_t kU1 = 384, kU2 = 416;    // U^T parts, 64 t packed in 32 columns
constexpr uint32_t kUd1 = 448, kUd2 = 480;  // (U^T diag(dec)) parts
constexpr uint32_t kCols = 512;
}  // namespace tcol

// mbarriers: the two [K;Q] copies, the V copy, and the products, each of
// which commits on its own so that its consumer waits for it alone: phase A's
// U part (A) and its Oi part (OI), [K;Q] K^T (D1), phase B (B), MMA2's W^T
// part (M2W) and its Ut^T part (M2).
enum { BKQ0 = 0, BKQ1 = 1, BV = 2, BA = 3, BD1 = 4, BB = 5, BM2 = 6, BOI = 7, BM2W = 8, kBars = 9 };

// x0 and x1 rounded to nearest-even bf16, packed with x0 in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float x0, float x1) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(x1), "f"(x0));
    return d;
}

// Two-term bf16 split of 8 consecutive values: hi = bf16(x), lo = bf16(x - hi),
// each packed as four pairs.
__device__ __forceinline__ void split8(const float *x, uint32_t (&hi)[4], uint32_t (&lo)[4]) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        hi[p] = pack_bf16x2(x[2 * p], x[2 * p + 1]);
        lo[p] = pack_bf16x2(x[2 * p] - __uint_as_float(hi[p] << 16),
                            x[2 * p + 1] - __uint_as_float(hi[p] & 0xffff0000u));
    }
}
__device__ __forceinline__ void st16(unsigned char *p, const uint32_t (&w)[4]) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void __launch_bounds__(kThreads, 1) gdn_prefill_kernel(const __grid_constant__ PrefArgs a) {
    const int h = blockIdx.x % a.h_v;
    const int seq = a.order[blockIdx.x / a.h_v];  // longest sequences first
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
    const int nch = (len + kC - 1) / kC;
    // Warps 0..15 hold the state and do the element-wise and triangular work
    // (4 warps per tensor-memory lane quadrant); warp 16 (lane 0) issues the
    // tensor copies and the tensor-core products, so that a product's issue
    // (which holds the issuing warp until the product queue has room) never
    // holds back the element-wise work.
    const bool ctl = warp == kCtl;
    const bool issuer = ctl && lane == 0;
    const int q4 = warp & 3, cq = (warp >> 2) & 3;  // lane quadrant, column quarter
    const int arow = 32 * q4 + lane;                // tensor-memory lane this thread reads
    const uint32_t lane_base = uint32_t(32 * q4) << 16;
    // This thread's share of S: row arow, columns 32cq .. 32cq+31.  Between
    // chunks S is held only as its two bf16 parts (the MMA operand tiles);
    // their sum carries about 17 significant bits, and since every chunk
    // scales the old state by e^{G_last}, the rounding does not accumulate.
    const size_t row_off = size_t(h) * kD * kD + size_t(arow) * kD + 32 * cq;
    auto load_s0 = [&](float (&v)[32]) {
        if (src >= 0) {
            const float4 *sp = reinterpret_cast<const float4 *>(a.pool + size_t(src) * a.slot_stride + row_off);
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const float4 w = sp[x];
                v[4 * x] = w.x;
                v[4 * x + 1] = w.y;
                v[4 * x + 2] = w.z;
                v[4 * x + 3] = w.w;
            }
        } else {
#pragma unroll
            for (int x = 0; x < 32; ++x) v[x] = 0.f;
        }
    };
    auto store_dst = [&](const float (&v)[32]) {
        float4 *dp = reinterpret_cast<float4 *>(a.pool + size_t(dst) * a.slot_stride + row_off);
#pragma unroll
        for (int x = 0; x < 8; ++x) dp[x] = make_float4(v[4 * x], v[4 * x + 1], v[4 * x + 2], v[4 * x + 3]);
    };
    if (nch == 0) {  // an empty sequence publishes its start state
        if (!ctl) {
            float v[32];
            load_s0(v);
            store_dst(v);
        }
        return;
    }

    extern __shared__ __align__(1024) unsigned char smraw[];
    const uint32_t raw_u = gdn::smem_u32(smraw);
    unsigned char *sm = smraw + (((raw_u + 1023u) & ~1023u) - raw_u);
    const uint32_t sb = gdn::smem_u32(sm);
    float *Af = reinterpret_cast<float *>(sm + smap::kX);
    float *Xs = reinterpret_cast<float *>(sm + smap::kScratch);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + smap::kBars);
    uint32_t *tbase = reinterpret_cast<uint32_t *>(sm + smap::kTbase);
    int *flags = reinterpret_cast<int *>(sm + smap::kFlags);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + smap::kAbort);
    auto vecp = [&](uint32_t base, int b) { return reinterpret_cast<float *>(sm + base + 256u * uint32_t(b)); };

    if (warp == 0) tc::tmem_alloc(tbase, tcol::kCols);
    if (tid == 0) {
        for (int b = 0; b < kBars; ++b) gdn::mbar_init(&bars[b], 1);
        *abort_flag = 0;
    }
    auto chunk_t0 = [&](int c) { return s0 + c * kC; };
    auto chunk_n = [&](int c) { return min(kC, len - c * kC); };
    // Raw g and beta of chunk c (0 past its tokens) by threads 64..127.
    auto load_gb = [&](int c, float &gr, float &br) {
        const int t = tid - 64;
        gr = br = 0.f;
        if (t < chunk_n(c)) {
            gr = a.g[size_t(chunk_t0(c) + t) * a.h_v + h];
            br = a.beta[size_t(chunk_t0(c) + t) * a.h_v + h];
        }
    };
    const bool gb_thread = tid >= 64 && tid < 128;
    if (gb_thread) {
        float gr, br;
        load_gb(0, gr, br);
        vecp(smap::kGraw, 0)[tid - 64] = gr;
        vecp(smap::kBraw, 0)[tid - 64] = br;
    }
    gdn::fence_proxy_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmb = *tbase;

    // Barrier bookkeeping.  `par` (the same in every thread) holds the parity
    // of each barrier's next phase; it advances at fixed points of the
    // schedule, after every waiter of that phase.  The issuer also keeps the
    // phases it started (`armed`, with their parities), which an early exit
    // still waits for before the shared and tensor memory are released.
    uint32_t par = 0, armed = 0, arm_par = 0, nwait = 0;
    // SIMT threads: thread 0 waits (bounded) for the barriers in `mask`, the
    // others learn the outcome; on success the phases are acquired.
    auto wait_simt = [&](uint32_t mask) {
        int *flag = flags + (nwait++ & 3u);
        if (tid == 0) {
            bool good = *abort_flag == 0;
            for (int b = 0; b < kBars; ++b)
                if (good && ((mask >> b) & 1u)) good = gdn::mbar_wait_bounded(&bars[b], (par >> b) & 1u, a.wait_ns);
            if (!good) *abort_flag = 1;
            *flag = good ? 1 : 0;
        }
        simt_sync();
        const bool good = *flag != 0;
        if (good) {
            for (int b = 0; b < kBars; ++b)
                if ((mask >> b) & 1u) (void)gdn::mbar_try_wait(&bars[b], (par >> b) & 1u);
            tc::fence_after();
        }
        return good;
    };
    // The issuer waits (bounded) for one barrier before a product or a copy
    // that depends on it.
    auto ctl_wait = [&](int b) {
        if (*abort_flag) return false;
        if (gdn::mbar_wait_bounded(&bars[b], (par >> b) & 1u, a.wait_ns)) return true;
        *abort_flag = 1;
        return false;
    };
    auto arm = [&](int b) {
        armed |= 1u << b;
        arm_par = (arm_par & ~(1u << b)) | (par & (1u << b));
    };

    // Tensor copies (issuer).
    auto issue_kq = [&](int c, int b) {
        uint64_t *bar = &bars[BKQ0 + b];
        gdn::mbar_arrive_expect_tx(bar, 32768u);
        arm(BKQ0 + b);
        if (a.withhold && c == nch - 1) return;  // self-test: this phase never completes
        unsigned char *d = sm + smap::kKQ + 32768u * uint32_t(b);
#pragma unroll
        for (int at = 0; at < 2; ++at) {
            gdn::tma_load_3d(d + at * 16384, &a.tm_k, 64 * at, hq, chunk_t0(c), bar);
            gdn::tma_load_3d(d + at * 16384 + 8192, &a.tm_q, 64 * at, hq, chunk_t0(c), bar);
        }
    };
    auto issue_v = [&](int c) {
        gdn::mbar_arrive_expect_tx(&bars[BV], 16384u);
        arm(BV);
#pragma unroll
        for (int at = 0; at < 2; ++at) gdn::tma_load_3d(sm + smap::kV + at * 8192, &a.tm_v, 64 * at, h, chunk_t0(c), &bars[BV]);
    };
    // Rows n..63 of a partial chunk's tiles hold the next sequence's rows or
    // padding: zeroed once the copy has landed, before a product reads them.
    auto zero_kq_rows = [&](int b, int n) {
        unsigned char *d = sm + smap::kKQ + 32768u * uint32_t(b);
        for (int e = tid; e < (kC - n) * 32; e += kSimt) {
            const int row = n + (e >> 5), piece = e & 31, which = piece >> 3;
            *reinterpret_cast<uint4 *>(d + (which & 1) * 16384 + (which >> 1) * 8192 + row * 128 + (piece & 7) * 16) =
                make_uint4(0, 0, 0, 0);
        }
    };
    auto zero_v_rows = [&](int n) {
        for (int e = tid; e < (kC - n) * 16; e += kSimt) {
            const int row = n + (e >> 4), piece = e & 15;
            *reinterpret_cast<uint4 *>(sm + smap::kV + (piece >> 3) * 8192 + row * 128 + (piece & 7) * 16) =
                make_uint4(0, 0, 0, 0);
        }
    };

    // Products (issuer).
    const uint64_t dsc = tc::smem_desc(sb);  // descriptor of any K-major tile: tc::desc_at(dsc, offset)
    auto kq_off = [](int b) { return smap::kKQ + 32768u * uint32_t(b); };
    // Phase A of the chunk of parity b: U^T += -S W^T (its consumer, the U
    // split, comes next).  Oi = S Q^T, needed only for the outputs, is issued
    // on its own after phase B.
    auto issue_phase_a_u = [&]() {
        constexpr uint32_t idU = tc::idesc_bf16(128, 64) | tc::kBMnMajor | tc::kNegA;
        const uint64_t w1b = tc::smem_desc_mn(sb + smap::kW1, 8192), w2b = tc::smem_desc_mn(sb + smap::kW2, 8192);
#pragma unroll
        for (int at = 0; at < 2; ++at)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint32_t ka = at * 16384 + s * 32;
                const uint64_t a1 = tc::desc_at(dsc, smap::kS1 + ka), a2 = tc::desc_at(dsc, smap::kS2 + ka);
                const uint32_t wr = at * 8192 + s * 2048;  // rows d = 64 at + 16 s of the MN-major W tiles
                const uint64_t w1 = tc::desc_at(w1b, wr), w2 = tc::desc_at(w2b, wr);
                tc::mma_bf16(tmb + tcol::kU, a1, w1, idU, 1u);
                tc::mma_bf16(tmb + tcol::kU, a1, w2, idU, 1u);
                tc::mma_bf16(tmb + tcol::kU, a2, w1, idU, 1u);
            }
        tc::commit(&bars[BA]);
        arm(BA);
    };
    auto issue_phase_a_o = [&](int b) {
        constexpr uint32_t idO = tc::idesc_bf16(128, 64);
#pragma unroll
        for (int at = 0; at < 2; ++at)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint32_t ka = at * 16384 + s * 32;
                const uint64_t a1 = tc::desc_at(dsc, smap::kS1 + ka), a2 = tc::desc_at(dsc, smap::kS2 + ka);
                const uint64_t qd = tc::desc_at(dsc, kq_off(b) + at * 16384 + 8192 + s * 32);
                tc::mma_bf16(tmb + tcol::kOi, a1, qd, idO, (at | s) ? 1u : 0u);
                tc::mma_bf16(tmb + tcol::kOi, a2, qd, idO, 1u);
            }
        tc::commit(&bars[BOI]);
        arm(BOI);
    };
    auto issue_mma1 = [&](int b) {  // [K;Q] K^T of the chunk in buffer b
        constexpr uint32_t id1 = tc::idesc_bf16(128, 64);
#pragma unroll
        for (int at = 0; at < 2; ++at)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t d = tc::desc_at(dsc, kq_off(b) + at * 16384 + s * 32);
                tc::mma_bf16(tmb + tcol::kD1, d, d, id1, (at | s) ? 1u : 0u);
            }
        tc::commit(&bars[BD1]);
        arm(BD1);
    };
    auto issue_phase_b = [&](int b) {  // Oa = U^T P^T, dS = (U^T diag(dec)) K, A operands in tensor memory
        constexpr uint32_t idOa = tc::idesc_bf16(128, 64);
        constexpr uint32_t idS = tc::idesc_bf16(128, 128) | tc::kBMnMajor;
        const uint32_t pofs = smap::kP + 16384u * uint32_t(b);
        const uint64_t kmb = tc::smem_desc_mn(sb + kq_off(b), 16384);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const uint64_t p1 = tc::desc_at(dsc, pofs + s * 32), p2 = tc::desc_at(dsc, pofs + 8192 + s * 32);
            const uint64_t kmn = tc::desc_at(kmb, s * 2048);
            const uint32_t c8 = 8u * uint32_t(s);
            tc::mma_bf16_ts(tmb + tcol::kdS, tmb + tcol::kUd1 + c8, kmn, idS, s ? 1u : 0u);
            tc::mma_bf16_ts(tmb + tcol::kOa, tmb + tcol::kU1 + c8, p1, idOa, s ? 1u : 0u);
            tc::mma_bf16_ts(tmb + tcol::kdS, tmb + tcol::kUd2 + c8, kmn, idS, 1u);
            tc::mma_bf16_ts(tmb + tcol::kOa, tmb + tcol::kU1 + c8, p2, idOa, 1u);
            tc::mma_bf16_ts(tmb + tcol::kOa, tmb + tcol::kU2 + c8, p1, idOa, 1u);
        }
        tc::commit(&bars[BB]);
        arm(BB);
    };
    // MMA2 of the chunk in buffer b (A operands MN-major), W^T first (the W
    // split waits for it alone), then Ut^T into the U accumulator (the next
    // phase A, issued after it, accumulates onto it).
    auto issue_mma2 = [&](int b) {
        constexpr uint32_t id2 = tc::idesc_bf16(128, 64) | tc::kAMnMajor;
        const uint64_t ktb = tc::smem_desc_mn(sb + kq_off(b), 16384), vtb = tc::smem_desc_mn(sb + smap::kV, 8192);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const uint64_t kt = tc::desc_at(ktb, s * 2048);
            tc::mma_bf16(tmb + tcol::kD1, kt, tc::desc_at(dsc, smap::kBW1 + s * 32), id2, s ? 1u : 0u);
            tc::mma_bf16(tmb + tcol::kD1, kt, tc::desc_at(dsc, smap::kBW2 + s * 32), id2, 1u);
        }
        tc::commit(&bars[BM2W]);
        arm(BM2W);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const uint64_t vt = tc::desc_at(vtb, s * 2048);
            tc::mma_bf16(tmb + tcol::kU, vt, tc::desc_at(dsc, smap::kBU1 + s * 32), id2, s ? 1u : 0u);
            tc::mma_bf16(tmb + tcol::kU, vt, tc::desc_at(dsc, smap::kBU2 + s * 32), id2, 1u);
        }
        tc::commit(&bars[BM2]);
        arm(BM2);
    };

    // SIMT steps.
    auto write_S = [&](const float (&v)[32]) {
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            uint32_t hi[4], lo[4];
            split8(v + 8 * x, hi, lo);
            const uint32_t off = tc::swz_off(128, arow, 32 * cq + 8 * x);
            st16(sm + smap::kS1 + off, hi);
            st16(sm + smap::kS2 + off, lo);
        }
    };
    // S (this thread's 32 values) = the sum of its two parts.
    auto read_S = [&](float (&v)[32]) {
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const uint32_t off = tc::swz_off(128, arow, 32 * cq + 8 * x);
            const uint4 hi = *reinterpret_cast<const uint4 *>(sm + smap::kS1 + off);
            const uint4 lo = *reinterpret_cast<const uint4 *>(sm + smap::kS2 + off);
            const uint32_t hw[4] = {hi.x, hi.y, hi.z, hi.w}, lw[4] = {lo.x, lo.y, lo.z, lo.w};
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                v[8 * x + 2 * p] = __uint_as_float(hw[p] << 16) + __uint_as_float(lw[p] << 16);
                v[8 * x + 2 * p + 1] = __uint_as_float(hw[p] & 0xffff0000u) + __uint_as_float(lw[p] & 0xffff0000u);
            }
        }
    };
    // U^T of chunk c -> bf16 parts of U^T and of U^T diag(dec), into tensor memory.
    auto split_u = [&](int b, const uint32_t (&ur)[16]) {
        const float *dec = vecp(smap::kDec, b);
        float u[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) u[x] = __uint_as_float(ur[x]);
        const uint32_t c8 = 8u * uint32_t(cq);
        uint32_t hh[8], ll[8];
        split8(u, *reinterpret_cast<uint32_t(*)[4]>(hh), *reinterpret_cast<uint32_t(*)[4]>(ll));
        split8(u + 8, *reinterpret_cast<uint32_t(*)[4]>(hh + 4), *reinterpret_cast<uint32_t(*)[4]>(ll + 4));
        tc::st8(tmb + lane_base + tcol::kU1 + c8, hh);
        tc::st8(tmb + lane_base + tcol::kU2 + c8, ll);
#pragma unroll
        for (int x = 0; x < 16; ++x) u[x] *= dec[16 * cq + x];
        split8(u, *reinterpret_cast<uint32_t(*)[4]>(hh), *reinterpret_cast<uint32_t(*)[4]>(ll));
        split8(u + 8, *reinterpret_cast<uint32_t(*)[4]>(hh + 4), *reinterpret_cast<uint32_t(*)[4]>(ll + 4));
        tc::st8(tmb + lane_base + tcol::kUd1 + c8, hh);
        tc::st8(tmb + lane_base + tcol::kUd2 + c8, ll);
        tc::st_wait();
    };
    // From [K;Q] K^T of chunk c (n tokens, parity b), passed in v16: A
    // (lanes 0..63, fp32, left in v16 for store_a) and P (lanes 64..127, bf16
    // parts to the P tiles of parity b).  Masked entries are selected to
    // zero, never multiplied (the products of rows past n are finite, but not
    // necessarily zero).
    auto build_a_p = [&](int n, int b, float (&v16)[16]) {
        const float *G = vecp(smap::kG, b);
        const int t = arow & 63;
        const float gt = G[t];
        if (q4 < 2) {
            const float bt = vecp(smap::kBraw, b)[t];
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const int i = 16 * cq + x;
                const float e = chunkmath::gate_exp(gt - G[i]);
                v16[x] = (i < t && t < n) ? bt * e * v16[x] : 0.f;
            }
        } else {
            float pe[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const int i = 16 * cq + x;
                const float e = chunkmath::gate_exp(gt - G[i]);
                pe[x] = (i <= t && t < n) ? e * v16[x] : 0.f;
            }
            const uint32_t pofs = smap::kP + 16384u * uint32_t(b);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t hi[4], lo[4];
                split8(pe + 8 * half, hi, lo);
                const uint32_t off = tc::swz_off(64, t, 16 * cq + 8 * half);
                st16(sm + pofs + off, hi);
                st16(sm + pofs + 8192 + off, lo);
            }
        }
    };
    auto store_a = [&](const float (&v16)[16]) {
        if (q4 < 2) {
            const int t = arow & 63;
#pragma unroll
            for (int y = 0; y < 4; ++y)
                *reinterpret_cast<float4 *>(Af + t * kAs + 16 * cq + 4 * y) =
                    make_float4(v16[4 * y], v16[4 * y + 1], v16[4 * y + 2], v16[4 * y + 3]);
        }
    };
    // T -> T diag(beta e^G) and T diag(beta), bf16 parts (8 entries per thread).
    auto build_ab = [&](int b) {
        const int t = tid >> 3, i0 = (tid & 7) * 8;
        const float4 t0v = *reinterpret_cast<const float4 *>(Af + t * kAs + i0);
        const float4 t1v = *reinterpret_cast<const float4 *>(Af + t * kAs + i0 + 4);
        simt_sync();  // every T entry is read before the tiles overwrite it
        const float tv[8] = {t0v.x, t0v.y, t0v.z, t0v.w, t1v.x, t1v.y, t1v.z, t1v.w};
        const float *bt = vecp(smap::kBraw, b), *eg = vecp(smap::kEG, b);
        float xb[8], xv[8];
#pragma unroll
        for (int y = 0; y < 8; ++y) {
            xv[y] = tv[y] * bt[i0 + y];
            xb[y] = xv[y] * eg[i0 + y];
        }
        uint32_t bh[4], bl[4], vh[4], vl[4];
        split8(xb, bh, bl);
        split8(xv, vh, vl);
        const uint32_t off = tc::swz_off(64, t, i0);
        st16(sm + smap::kBW1 + off, bh);
        st16(sm + smap::kBW2 + off, bl);
        st16(sm + smap::kBU1 + off, vh);
        st16(sm + smap::kBU2 + off, vl);
    };
    // W^T (lanes d_k, columns t) -> the MN-major W parts.  W1 covers the
    // T diag(beta e^G) tiles, free once W^T is done; W2 covers the
    // T diag(beta) tiles, which MMA2's Ut^T half reads until all of MMA2 is
    // done, so the second parts are written after that wait.  All SIMT
    // threads call it (it waits); false if a wait ran out.
    auto split_w = [&]() {
        float w[16];
        tc::ld16(tmb + lane_base + tcol::kD1 + 16 * cq, w);
        uint32_t hi[2][4], lo[2][4];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            split8(w + 8 * half, hi[half], lo[half]);
            st16(sm + smap::kW1 + tc::swz_off(128, arow, 16 * cq + 8 * half), hi[half]);
        }
        if (!wait_simt(1u << BM2)) return false;
#pragma unroll
        for (int half = 0; half < 2; ++half) st16(sm + smap::kW2 + tc::swz_off(128, arow, 16 * cq + 8 * half), lo[half]);
        return true;
    };
    // Chunk c (parity b): S <- e^{G_last} S + dS.
    auto update_S = [&](int c, int b) {
        const int n = chunk_n(c);
        const float *eG = vecp(smap::kEG, b);
        const float egl = eG[n - 1];
        uint32_t d0[16], d1[16];
        tc::ld16_async(tmb + lane_base + tcol::kdS + uint32_t(32 * cq), d0);
        tc::ld16_async(tmb + lane_base + tcol::kdS + uint32_t(32 * cq + 16), d1);
        float sv[32];
        read_S(sv);
        tc::ld_wait();
        tc::ld_fence_regs(d0);
        tc::ld_fence_regs(d1);
#pragma unroll
        for (int x = 0; x < 16; ++x) {
            sv[x] = fmaf(egl, sv[x], __uint_as_float(d0[x]));
            sv[16 + x] = fmaf(egl, sv[16 + x], __uint_as_float(d1[x]));
        }
        write_S(sv);
    };
    // The outputs of chunk c (parity b), o = q_scale (e^G Oi + Oa), staged
    // as bf16 [t][d_v] in the chunk's P tiles (their last reader, phase B, is
    // done) and written as 16-byte rows.  They run at the start of the next
    // iteration, while phase A(c+1) executes (Oi and Oa are overwritten only
    // by that iteration's phase B and Oi, the P tiles only by its A/P build,
    // e^G only by its gate sums, all after the barrier that follows).
    auto outputs = [&](int c, int b) {
        const int n = chunk_n(c);
        const float *eG = vecp(smap::kEG, b);
        uint32_t oi[16], oa[16];
        tc::ld16_async(tmb + lane_base + tcol::kOi + uint32_t(16 * cq), oi);
        tc::ld16_async(tmb + lane_base + tcol::kOa + uint32_t(16 * cq), oa);
        tc::ld_wait();
        tc::ld_fence_regs(oi);
        tc::ld_fence_regs(oa);
        uint16_t *ostage = reinterpret_cast<uint16_t *>(sm + smap::kP + 16384u * uint32_t(b));
#pragma unroll
        for (int x = 0; x < 16; ++x) {
            const int t = 16 * cq + x;
            ostage[t * kD + arow] =
                gdn::f32_to_bf16(a.q_scale * fmaf(eG[t], __uint_as_float(oi[x]), __uint_as_float(oa[x])));
        }
        simt_sync();
        const int t0 = chunk_t0(c);
        for (int e = tid; e < n * 16; e += kSimt) {
            const int t = e >> 4, ch = e & 15;
            *reinterpret_cast<uint4 *>(a.o + (size_t(t0 + t) * a.h_v + h) * kD + ch * 8) =
                *reinterpret_cast<const uint4 *>(ostage + t * kD + ch * 8);
        }
    };

    if (issuer) {
        issue_kq(0, 0);
        issue_v(0);
        if (nch > 1) issue_kq(1, 1);
    }
    // Iteration c runs the scan of chunk c (c >= 0) beside the producer of
    // chunk c+1 (c+1 < nch); c = -1 only produces chunk 0 and stages S.
    bool ok = true;
    for (int c = -1; c < nch; ++c) {
        const bool scan = c >= 0, prod = c + 1 < nch, next2 = c + 2 < nch;
        const int sbuf = c & 1, pbuf = (c + 1) & 1;
        const int np = prod ? chunk_n(c + 1) : 0;
        const bool partial = prod && np < kC;
        // ---- slot 1: phase A(c); MMA1(c+1); the outputs of chunk c-1; G, e^G,
        // dec of chunk c+1; raw g, beta of chunk c+2
        if (issuer && scan) issue_phase_a_u();
        if (partial) {
            // the partial last chunk: its K and Q rows past n become zero first
            if (!ctl && wait_simt(1u << (BKQ0 + pbuf))) {
                zero_kq_rows(pbuf, np);
                gdn::fence_proxy_async_smem();
            }
            __syncthreads();
            if (*abort_flag) {
                ok = false;
                break;
            }
            if (issuer) issue_mma1(pbuf);
        } else if (prod && issuer) {
            if (ctl_wait(BKQ0 + pbuf)) issue_mma1(pbuf);
        }
        float gr = 0.f, br = 0.f;
        bool good = true;
        if (!ctl) {
            if (c >= 1) {  // the outputs of chunk c-1 while phase A(c) executes
                outputs(c - 1, pbuf);
                simt_sync();  // e^G of chunk c-1 is read before the gate sums below rewrite it
            }
            if (prod && warp == 1) {
                float *G = vecp(smap::kG, pbuf);
                chunkmath::chunk_cumsum(vecp(smap::kGraw, pbuf), np, G);
                __syncwarp();
                const float gl = G[np - 1];
                for (int e = lane; e < kC; e += 32) {
                    const float ge = G[e];
                    vecp(smap::kEG, pbuf)[e] = expf(ge);
                    vecp(smap::kDec, pbuf)[e] = e < np ? expf(gl - ge) : 0.f;
                }
            }
            if (next2 && gb_thread) load_gb(c + 2, gr, br);
            good = wait_simt((scan ? 1u << BA : 0u) | (prod ? 1u << BD1 : 0u));
            // ---- slot 2: U parts of chunk c; A and P of chunk c+1
            if (good) {
                if (prod) {
                    uint32_t vr[16];
                    tc::ld16_async(tmb + lane_base + tcol::kD1 + 16 * cq, vr);
                    tc::ld_wait();
                    tc::ld_fence_regs(vr);
                    float av[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) av[x] = __uint_as_float(vr[x]);
                    build_a_p(np, pbuf, av);
                    store_a(av);
                }
                if (scan) {
                    uint32_t ur[16];
                    tc::ld16_async(tmb + lane_base + tcol::kU + 16 * cq, ur);
                    tc::ld_wait();
                    tc::ld_fence_regs(ur);
                    split_u(sbuf, ur);
                }
                gdn::fence_proxy_async_smem();
                tc::fence_before();
            }
        }
        par ^= (scan ? 1u << BA : 0u) | (prod ? (1u << BD1) | (1u << (BKQ0 + pbuf)) : 0u);
        __syncthreads();
        if (*abort_flag) {
            ok = false;
            break;
        }
        // ---- slot 3: phase B(c) beside T of chunk c+1 and its operands
        if (issuer && scan) {
            tc::fence_after();
            issue_phase_b(sbuf);
            issue_phase_a_o(sbuf);  // Oi(c), after the outputs of chunk c-1 have read Oi(c-1)
        }
        if (!ctl && prod) {
            chunkmath::solve_unit_lower<kSimt, kAs>(Af, Xs, tid, [] { simt_sync(); });
            build_ab(pbuf);
            if (partial && wait_simt(1u << BV)) zero_v_rows(np);
            gdn::fence_proxy_async_smem();
            tc::fence_before();
        }
        __syncthreads();
        if (*abort_flag) {
            ok = false;
            break;
        }
        // ---- slot 4: MMA2(c+1); update and outputs of chunk c; W parts of
        // chunk c+1; chunk c+2's K, Q (once phase B(c) is done) and V (once MMA2 is)
        if (issuer) {
            tc::fence_after();
            if (prod && (partial || ctl_wait(BV))) issue_mma2(pbuf);
            if (scan && next2 && ctl_wait(BB) && ctl_wait(BOI)) issue_kq(c + 2, sbuf);
            if (prod && next2 && ctl_wait(BM2)) issue_v(c + 2);
        }
        if (!ctl) {
            good = true;
            if (scan) {
                good = wait_simt((1u << BB) | (1u << BOI));
                if (good) update_S(c, sbuf);
            } else {
                float v[32];
                load_s0(v);
                write_S(v);
            }
            if (prod && good && wait_simt(1u << BM2W)) (void)split_w();
            if (next2 && gb_thread) {
                vecp(smap::kGraw, sbuf)[tid - 64] = gr;
                vecp(smap::kBraw, sbuf)[tid - 64] = br;
            }
            gdn::fence_proxy_async_smem();
            tc::fence_before();
        }
        par ^= (scan ? (1u << BB) | (1u << BOI) : 0u) | (prod ? (1u << BM2) | (1u << BM2W) | (1u << BV) : 0u);
        __syncthreads();
        if (*abort_flag) {
            ok = false;
            break;
        }
        tc::fence_after();
    }
    if (!ok) {
        // A wait ran out: wait (again bounded) for whatever is still in
        // flight into this CTA's shared or tensor memory, report, and leave
        // the destination slot untouched.
        if (issuer) {
            for (int b = 0; b < kBars; ++b)
                if ((armed >> b) & 1u) (void)gdn::mbar_wait_bounded(&bars[b], (arm_par >> b) & 1u, a.wait_ns);
            gdn::set_status(a.status, GDN_DEV_TIMEOUT);
        }
    } else if (!ctl) {
        outputs(nch - 1, (nch - 1) & 1);  // the last chunk's outputs
        if (!a.status || !(*reinterpret_cast<volatile uint32_t *>(a.status) & GDN_DEV_TIMEOUT)) {
            // Publication: only the final state, and not after any bounded
            // wait (here or in an earlier launch) has run out.
            float v[32];
            read_S(v);
            store_dst(v);
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmb, tcol::kCols);
}

// order[r] = the sequence with the r-th largest length (ties by index), so
// that the longest dependency chains start in the first wave.  One block.
__global__ void gdn_prefill_order_kernel(const int32_t *cu, int nseq, int32_t *order) {
    for (int i = threadIdx.x; i < nseq; i += blockDim.x) {
        const int li = cu[i + 1] - cu[i];
        int r = 0;
        for (int j = 0; j < nseq; ++j) {
            const int lj = cu[j + 1] - cu[j];
            r += (lj > li || (lj == li && j < i)) ? 1 : 0;
        }
        order[r] = i;
    }
}

}  // namespace

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

// Workspace: the length order of the sequences (nseq int32).
extern "C" size_t gdn_prefill_workspace_bytes(const gdn_dims *dims, int32_t nseq, int32_t row_capacity) {
    if (!dims || nseq < 0 || row_capacity < 0) return 0;
    return align16(size_t(nseq) * 4);
}

// d in {16, 32, 64}: the fp32 chunk-form kernel (gdn_prefill_small.cu).
int gdn_prefill_small_launch(const gdn_dims *dims, int32_t nseq, int32_t row_capacity, const int32_t *cu_seqlens,
                             const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v, const float *g,
                             const float *beta, float *pool_layer, int64_t slot_stride, int32_t num_slots,
                             const int32_t *src_slot, const int32_t *dst_slot, gdn_bf16 *o, const int32_t *order,
                             uint32_t *dev_status, cudaStream_t st);

static int prefill_launch(const gdn_dims *dims, int32_t nseq, int32_t row_capacity, const int32_t *cu_seqlens,
                          int32_t max_seqlen, const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                          const float *g, const float *beta, float *pool_layer, int64_t slot_stride,
                          int32_t num_slots, const int32_t *src_slot, const int32_t *dst_slot, gdn_bf16 *o,
                          int32_t chunk, void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                          uint64_t wait_ns, int withhold, void *stream) {
    if (!dims) return GDN_ERR_NULL;
    if (!gdn_host::dims_ok(dims)) return GDN_ERR_SHAPE;
    if (withhold && dims->d_k != kD) return GDN_ERR_SHAPE;  // the self-test needs the copy engine's path
    if (chunk != kC) return GDN_ERR_ARG;
    if (nseq < 0 || row_capacity < 0 || max_seqlen < 0 || num_slots <= 0) return GDN_ERR_ARG;
    if (nseq == 0) return GDN_OK;
    if (!cu_seqlens || !q || !k || !v || !g || !beta || !pool_layer || !src_slot || !dst_slot || !o)
        return GDN_ERR_NULL;
    const int64_t se = int64_t(dims->h_v) * dims->d_v * dims->d_k;
    if (slot_stride < se || (slot_stride % 4) != 0) return GDN_ERR_ARG;
    if (!gdn_host::aligned16(pool_layer) || !gdn_host::aligned16(q) || !gdn_host::aligned16(k) ||
        !gdn_host::aligned16(v) || !gdn_host::aligned16(o))
        return GDN_ERR_ARG;
    const size_t need = gdn_prefill_workspace_bytes(dims, nseq, row_capacity);
    if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE;
    if (!gdn_host::aligned16(workspace)) return GDN_ERR_ARG;
    const long long grid = (long long)nseq * dims->h_v;
    if (grid > 0x7fffffffLL) return GDN_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dims->d_k != kD) {
        gdn_prefill_order_kernel<<<1, 256, 0, st>>>(cu_seqlens, nseq, static_cast<int32_t *>(workspace));
        if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
        return gdn_prefill_small_launch(dims, nseq, row_capacity, cu_seqlens, q, k, v, g, beta, pool_layer,
                                        slot_stride, num_slots, src_slot, dst_slot, o,
                                        static_cast<const int32_t *>(workspace), dev_status, st);
    }
    PrefArgs a{};
    a.cu = cu_seqlens;
    a.nseq = nseq;
    a.h_qk = dims->h_qk;
    a.h_v = dims->h_v;
    a.grp = dims->h_v / dims->h_qk;
    a.row_capacity = row_capacity;
    a.num_slots = num_slots;
    a.g = g;
    a.beta = beta;
    a.pool = pool_layer;
    a.slot_stride = slot_stride;
    a.src_slot = src_slot;
    a.dst_slot = dst_slot;
    a.o = o;
    a.order = static_cast<const int32_t *>(workspace);
    a.q_scale = dims->q_scale;
    a.status = dev_status;
    a.wait_ns = wait_ns;
    a.withhold = withhold;
    if (!encode_rows(&a.tm_q, q, dims->h_qk, row_capacity) || !encode_rows(&a.tm_k, k, dims->h_qk, row_capacity) ||
        !encode_rows(&a.tm_v, v, dims->h_v, row_capacity))
        return GDN_ERR_CUDA;
    if (cudaFuncSetAttribute(gdn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smap::kSmem)) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    gdn_prefill_order_kernel<<<1, 256, 0, st>>>(cu_seqlens, nseq, static_cast<int32_t *>(workspace));
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    gdn_prefill_kernel<<<unsigned(grid), kThreads, smap::kSmem, st>>>(a);
    return gdn_host::launch_status(cudaGetLastError());
}

extern "C" int gdn_chunked_prefill(const gdn_dims *dims, int32_t nseq, int32_t row_capacity,
                                   const int32_t *cu_seqlens, int32_t max_seqlen, const gdn_bf16 *q,
                                   const gdn_bf16 *k, const gdn_bf16 *v, const float *g, const float *beta,
                                   float *pool_layer, int64_t slot_stride, int32_t num_slots,
                                   const int32_t *src_slot, const int32_t *dst_slot, gdn_bf16 *o, int32_t chunk,
                                   void *workspace, size_t workspace_bytes, uint32_t *dev_status, void *stream) {
    return prefill_launch(dims, nseq, row_capacity, cu_seqlens, max_seqlen, q, k, v, g, beta, pool_layer,
                          slot_stride, num_slots, src_slot, dst_slot, o, chunk, workspace, workspace_bytes,
                          dev_status, gdn::kWaitLimitNs, 0, stream);
}

extern "C" int gdn_selftest_prefill_timeout(const gdn_dims *dims, int32_t nseq, int32_t row_capacity,
                                            const int32_t *cu_seqlens, const gdn_bf16 *q, const gdn_bf16 *k,
                                            const gdn_bf16 *v, const float *g, const float *beta,
                                            float *pool_layer, int64_t slot_stride, int32_t num_slots,
                                            const int32_t *src_slot, const int32_t *dst_slot, gdn_bf16 *o,
                                            void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                                            uint64_t limit_ns, void *stream) {
    if (limit_ns == 0 || limit_ns > gdn::kWaitLimitNs) return GDN_ERR_ARG;
    return prefill_launch(dims, nseq, row_capacity, cu_seqlens, 0, q, k, v, g, beta, pool_layer, slot_stride,
                          num_slots, src_slot, dst_slot, o, kC, workspace, workspace_bytes, dev_status, limit_ns, 1,
                          stream);
}
