// Greedy target choice over the vocabulary and draft acceptance (sm_103a).
//
// Operation ("Native three-step MTP", Apply...: greedy requests; "Run chained
// MTP drafting in the batch Engine", Summary: device-resident draft ids and
// cumulative telemetry; Quality follow-up: verification-row selection and
// per-request bonus):
//   argmax[t]     = first index of the largest bf16 logit of row t
//   accept_len[r] = longest j with tokens[t0+i] == argmax[t0+i-1], i = 1..j
//   bonus[r]      = argmax[t0+j]
//
// Two launches.  (1) argmax_partial: rows x splits CTAs stream the logits
// with 16-byte loads and reduce a 64-bit key per split,
//     key = order17(value) << 32 | (0xffffffff - index),
// whose unsigned maximum is the largest value with the lowest index (order17
// maps bf16 to an order-preserving integer, -0 to +0, and every NaN above
// +inf so that the first NaN wins).  (2) accept_finalize: one warp per
// request reduces its rows' partial keys, applies the acceptance rule, writes
// the emitted tokens and adds to the telemetry counters.
// HBM roofline: vocab x 2 bytes per row read once.
#include "common.cuh"

namespace {

constexpr int kArgThreads = 256;
constexpr int kMaxSplits = 64;
constexpr int kMinSplitElems = 2048;

__device__ __forceinline__ uint32_t order17(uint32_t bits) {
    uint32_t m = bits & 0x7fffu;
    if (m > 0x7f80u) return 0x10000u;            // NaN
    if (m == 0) return 0x8000u;                  // +0 and -0
    return (bits & 0x8000u) ? (0x7fffu - m) : (0x8000u + m);
}

__device__ __forceinline__ unsigned long long make_key(uint32_t bits, uint32_t idx) {
    return (static_cast<unsigned long long>(order17(bits)) << 32) | (0xffffffffu - idx);
}

// Largest of two bf16 pairs, lane by lane, NaN if either is NaN.
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// order17 of the largest of the 8 bf16 values of a 16-byte vector.
__device__ __forceinline__ uint32_t vec_max_order(const uint4 &w) {
    const uint32_t m = bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w));
    const uint32_t lo = order17(m & 0xffffu), hi = order17(m >> 16);
    return lo > hi ? lo : hi;
}

// Running (order, index) of a thread's scan over increasing indices: a
// vector whose largest value does not beat the best so far is skipped with
// a few packed maxima; otherwise its first element of that order is found
// (ties keep the earlier index, so the first occurrence wins).
__device__ __forceinline__ void scan_vec(const uint4 &w, uint32_t base, uint32_t vo, uint32_t &best_o,
                                         uint32_t &best_i) {
    if (vo <= best_o) return;
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t bits = (e & 1) ? (ws[e >> 1] >> 16) : (ws[e >> 1] & 0xffffu);
        if (order17(bits) == vo) {
            best_o = vo;
            best_i = base + uint32_t(e);
            return;
        }
    }
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}

__device__ __forceinline__ unsigned long long warp_max64(unsigned long long x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x = umax64(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
}

struct ArgArgs {
    const int32_t *cu_rows;
    int32_t B, row_capacity, splits;
    const uint16_t *logits;
    int64_t vocab, row_stride, chunk;
    int vec;  // 16-byte loads allowed
    unsigned long long *partial;
};

__global__ void __launch_bounds__(kArgThreads) argmax_partial_kernel(const ArgArgs a) {
    gdn::pdl_enter();
    const int split = blockIdx.x;
    const int row = blockIdx.y;
    int total = a.cu_rows[a.B];
    if (total > a.row_capacity || total < 0) total = a.row_capacity;
    if (row >= total) return;
    const int64_t c0 = int64_t(split) * a.chunk;
    const int64_t c1 = min(a.vocab, c0 + a.chunk);
    const uint16_t *rp = a.logits + int64_t(row) * a.row_stride;
    unsigned long long best = 0ull;
    if (c1 <= c0) {
        // empty range: nothing to scan
    } else if (a.vec) {
        // c0 and chunk are multiples of 8 elements: whole 16-byte vectors.
        const uint4 *vp = reinterpret_cast<const uint4 *>(rp + c0);
        const int64_t nvec = (c1 - c0) / 8;
        int64_t i = threadIdx.x;
        const int lane = threadIdx.x & 31;
        uint32_t best_o = 0, best_i = 0;  // order 0 is below every value: nothing seen yet
        // The warp's prefilter: the order of the largest value any of its lanes
        // has recorded.  A group of 4 kArgThreads vectors (indices above every
        // earlier group's) whose largest value does not exceed it can neither
        // beat that value nor win a tie with it, so the whole warp skips the
        // exact scan; the test is the same for every lane (one warp-wide max),
        // so the warp never runs the scan for one lane's sake.  The loop runs
        // while the warp's last lane has a whole group, so it is uniform too,
        // and the next group's loads go out before this group is examined.
        uint32_t warp_best = 0;
        bool have = i - lane + 31 + 3 * kArgThreads < nvec;
        uint4 w[4];
        if (have) {
#pragma unroll
            for (int u = 0; u < 4; ++u) w[u] = __ldcs(vp + i + u * kArgThreads);
        }
        while (have) {
            const int64_t inext = i + 4 * kArgThreads;
            const bool more = inext - lane + 31 + 3 * kArgThreads < nvec;
            uint4 nx[4];
            if (more) {
#pragma unroll
                for (int u = 0; u < 4; ++u) nx[u] = __ldcs(vp + inext + u * kArgThreads);
            }
            uint32_t m = bmax2(bmax2(bmax2(w[0].x, w[0].y), bmax2(w[0].z, w[0].w)),
                               bmax2(bmax2(w[1].x, w[1].y), bmax2(w[1].z, w[1].w)));
            m = bmax2(m, bmax2(bmax2(bmax2(w[2].x, w[2].y), bmax2(w[2].z, w[2].w)),
                               bmax2(bmax2(w[3].x, w[3].y), bmax2(w[3].z, w[3].w))));
            const uint32_t mo_lo = order17(m & 0xffffu), mo_hi = order17(m >> 16);
            const uint32_t wm = __reduce_max_sync(0xffffffffu, mo_lo > mo_hi ? mo_lo : mo_hi);
            if (wm > warp_best) {
                warp_best = wm;
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    scan_vec(w[u], uint32_t(c0 + (i + u * kArgThreads) * 8), vec_max_order(w[u]), best_o, best_i);
            }
            i = inext;
            have = more;
            if (more) {
#pragma unroll
                for (int u = 0; u < 4; ++u) w[u] = nx[u];
            }
        }
        for (; i < nvec; i += kArgThreads) {
            const uint4 w = __ldcs(vp + i);
            scan_vec(w, uint32_t(c0 + i * 8), vec_max_order(w), best_o, best_i);
        }
        if (best_o) best = (static_cast<unsigned long long>(best_o) << 32) | (0xffffffffu - best_i);
        // tail (vocab not a multiple of 8)
        for (int64_t j = c0 + nvec * 8 + threadIdx.x; j < c1; j += kArgThreads)
            best = umax64(best, make_key(rp[j], uint32_t(j)));
    } else {
        for (int64_t j = c0 + threadIdx.x; j < c1; j += kArgThreads) best = umax64(best, make_key(rp[j], uint32_t(j)));
    }
    __shared__ unsigned long long red[kArgThreads / 32];
    best = warp_max64(best);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x < 32) {
        unsigned long long x = threadIdx.x < kArgThreads / 32 ? red[threadIdx.x] : 0ull;
        x = warp_max64(x);
        if (threadIdx.x == 0) a.partial[int64_t(row) * a.splits + split] = x;
    }
}

struct AccArgs {
    const int32_t *cu_rows;
    int32_t B, row_capacity, splits;
    int64_t vocab;
    const unsigned long long *partial;
    const int32_t *tokens;
    int32_t *argmax, *accept_len, *bonus, *out_tokens;
    mtp_stats *stats;
    uint32_t *status;
};

constexpr int kAccWarps = 4;

__global__ void __launch_bounds__(kAccWarps * 32) accept_finalize_kernel(const AccArgs a) {
    gdn::pdl_enter();
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * kAccWarps + (threadIdx.x >> 5);
    if (r >= a.B) return;
    if (r == 0 && lane == 0 && a.stats) atomicAdd(reinterpret_cast<unsigned long long *>(&a.stats->steps), 1ull);
    const int t0 = a.cu_rows[r];
    const int t1 = a.cu_rows[r + 1];
    const int n = t1 - t0;
    // rows past cu_rows[B] got no partial maxima (non-monotone table)
    const int total = a.cu_rows[a.B];
    if (t0 < 0 || n < 1 || n > GDN_MAX_ROWS || t1 > a.row_capacity || t1 > total) {
        if (lane == 0) {
            gdn::set_status(a.status, GDN_DEV_ROWS_BAD);
            a.accept_len[r] = -1;
            a.bonus[r] = -1;
        }
        return;
    }
    int am[GDN_MAX_ROWS];
#pragma unroll
    for (int m = 0; m < GDN_MAX_ROWS; ++m) {
        if (m < n) {
            unsigned long long x = 0ull;
            for (int s = lane; s < a.splits; s += 32) x = umax64(x, a.partial[int64_t(t0 + m) * a.splits + s]);
            x = warp_max64(x);
            am[m] = x == 0ull ? -1 : int(0xffffffffu - uint32_t(x & 0xffffffffull));
        }
    }
    if (lane != 0) return;
    const int K = n - 1;
    bool oor = false;
    for (int i = 1; i <= K; ++i) {
        const int d = a.tokens[t0 + i];
        if (d < 0 || int64_t(d) >= a.vocab) oor = true;
    }
    int j = 0;
    while (j < K && a.tokens[t0 + j + 1] == am[j]) ++j;
    for (int m = 0; m < n; ++m) {
        a.argmax[t0 + m] = am[m];
        a.out_tokens[t0 + m] = m <= j ? am[m] : -1;
    }
    a.accept_len[r] = j;
    a.bonus[r] = am[j];
    if (oor) gdn::set_status(a.status, GDN_DEV_TOKEN_OOR);
    if (a.stats) {
        atomicAdd(reinterpret_cast<unsigned long long *>(&a.stats->proposed), (unsigned long long)K);
        atomicAdd(reinterpret_cast<unsigned long long *>(&a.stats->evaluated),
                  (unsigned long long)(j + 1 < K ? j + 1 : K));
        atomicAdd(reinterpret_cast<unsigned long long *>(&a.stats->accepted), (unsigned long long)j);
        atomicAdd(reinterpret_cast<unsigned long long *>(&a.stats->emitted), (unsigned long long)(j + 1));
    }
}

// Vocabulary splits per row: about 1024 CTAs in all, at most kMaxSplits and
// at least kMinSplitElems entries each.
int accept_splits(int32_t rows, int64_t vocab) {
    int64_t s = (1024 + int64_t(rows > 0 ? rows : 1) - 1) / int64_t(rows > 0 ? rows : 1);
    if (s > kMaxSplits) s = kMaxSplits;
    int64_t smax = vocab / kMinSplitElems;
    if (smax < 1) smax = 1;
    if (s > smax) s = smax;
    if (s < 1) s = 1;
    return int(s);
}

}  // namespace

int gdn_accept_launch(int32_t B, int32_t row_capacity, const int32_t *cu_rows, const gdn_bf16 *logits,
                      int64_t vocab, int64_t row_stride, const int32_t *tokens, int32_t *argmax,
                      int32_t *accept_len, int32_t *bonus, int32_t *out_tokens, mtp_stats *stats,
                      void *workspace, size_t workspace_bytes, uint32_t *dev_status, cudaStream_t st);

extern "C" size_t mtp_accept_workspace_bytes(int32_t row_capacity, int64_t vocab) {
    if (row_capacity <= 0 || vocab <= 0) return 0;
    return size_t(row_capacity) * size_t(accept_splits(row_capacity, vocab)) * sizeof(unsigned long long);
}

int gdn_accept_launch(int32_t B, int32_t row_capacity, const int32_t *cu_rows, const gdn_bf16 *logits,
                      int64_t vocab, int64_t row_stride, const int32_t *tokens, int32_t *argmax,
                      int32_t *accept_len, int32_t *bonus, int32_t *out_tokens, mtp_stats *stats,
                      void *workspace, size_t workspace_bytes, uint32_t *dev_status, cudaStream_t st) {
    if (B < 0 || row_capacity < 0 || vocab <= 0 || row_stride < vocab || vocab > 0x7fffffffLL) return GDN_ERR_ARG;
    if (!cu_rows || !logits || !tokens || !argmax || !accept_len || !bonus || !out_tokens) return GDN_ERR_NULL;
    if (B == 0) return GDN_OK;
    const size_t need = mtp_accept_workspace_bytes(row_capacity, vocab);
    if (row_capacity > 0 && (!workspace || workspace_bytes < need)) return GDN_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 7u) != 0) return GDN_ERR_ARG;
    const int splits = accept_splits(row_capacity, vocab);
    if (row_capacity > 0) {
        ArgArgs aa{};
        aa.cu_rows = cu_rows;
        aa.B = B;
        aa.row_capacity = row_capacity;
        aa.splits = splits;
        aa.logits = logits;
        aa.vocab = vocab;
        aa.row_stride = row_stride;
        int64_t chunk = (vocab + splits - 1) / splits;
        chunk = (chunk + 7) / 8 * 8;
        aa.chunk = chunk;
        aa.vec = (gdn_host::aligned16(logits) && (row_stride % 8) == 0) ? 1 : 0;
        aa.partial = static_cast<unsigned long long *>(workspace);
        if (row_capacity > 65535) return GDN_ERR_ARG;
        const int st_a = gdn_host::launch_pdl(argmax_partial_kernel, dim3(splits, row_capacity), dim3(kArgThreads), 0,
                                              st, aa);
        if (st_a != GDN_OK) return st_a;
    }
    AccArgs ac{};
    ac.cu_rows = cu_rows;
    ac.B = B;
    ac.row_capacity = row_capacity;
    ac.splits = splits;
    ac.vocab = vocab;
    ac.partial = static_cast<const unsigned long long *>(workspace);
    ac.tokens = tokens;
    ac.argmax = argmax;
    ac.accept_len = accept_len;
    ac.bonus = bonus;
    ac.out_tokens = out_tokens;
    ac.stats = stats;
    ac.status = dev_status;
    return gdn_host::launch_pdl(accept_finalize_kernel, dim3((B + kAccWarps - 1) / kAccWarps), dim3(kAccWarps * 32), 0,
                                st, ac);
}

extern "C" int mtp_greedy_accept(int32_t B, int32_t row_capacity, const int32_t *cu_rows, const gdn_bf16 *logits,
                                 int64_t vocab, int64_t row_stride, const int32_t *tokens, int32_t *argmax,
                                 int32_t *accept_len, int32_t *bonus, int32_t *out_tokens, mtp_stats *stats,
                                 void *workspace, size_t workspace_bytes, uint32_t *dev_status, void *stream) {
    return gdn_accept_launch(B, row_capacity, cu_rows, logits, vocab, row_stride, tokens, argmax, accept_len,
                             bonus, out_tokens, stats, workspace, workspace_bytes, dev_status,
                             static_cast<cudaStream_t>(stream));
}
