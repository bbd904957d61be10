// Commit / rollback of every layer's state slot to its accepted checkpoint
// (sm_103a).  "Run chained MTP drafting in the batch Engine", Correctness fix:
// a rejected request must publish the checkpoint of its accepted row and
// never one that the transaction did not write; RC4 evidence: rollback.
//
// One launch covers all (request, layer) pairs.  Each CTA copies one
// contiguous 32 KB piece of a state (fp32 [h_v][d_v][d_k]) with 16-byte
// streaming loads and stores, after checking the checkpoint tag written by
// gdn_verify: the tag must carry this transaction id and a row count larger
// than the accept length.  HBM roofline: read + write of S_bytes per pair.
#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kChunkFloats = 8192;  // 32 KB per CTA
constexpr int kUnroll = kChunkFloats / 4 / kThreads;

struct CommitArgs {
    int32_t B, L, row_capacity, num_slots, chunks;
    const int32_t *cu_rows, *accept_len, *dst_slot;
    const float *ckpt;
    int64_t ckpt_layer_stride, s_elems, slot_stride, layer_stride;
    const uint64_t *tag;
    uint32_t txn;
    float *pool;
    uint32_t *status;
    // set by the host driver: a request the transaction gate refused
    // (accept_len < 0, its cause already reported) is skipped silently
    int32_t gated;
};

__global__ void __launch_bounds__(kThreads) gdn_commit_kernel(const CommitArgs a) {
    gdn::pdl_enter();
    const long long idx = blockIdx.x;
    const int c = int(idx % a.chunks);
    const long long rl = idx / a.chunks;
    const int r = int(rl % a.B);
    const int l = int(rl / a.B);
    if (a.status && (*reinterpret_cast<volatile uint32_t *>(a.status) & GDN_DEV_TIMEOUT)) return;
    const uint64_t tag = a.tag[int64_t(l) * a.B + r];
    const int j = a.accept_len[r];
    const int dst = a.dst_slot[r];
    const int t0 = a.cu_rows[r];
    const uint32_t n = uint32_t(tag & 0xffffffffull);
    if (a.gated && j < 0) return;
    uint32_t bad = 0;
    if (uint32_t(tag >> 32) != a.txn || n == 0)
        bad = GDN_DEV_CKPT_UNWRITTEN;
    else if (j < 0 || uint32_t(j) >= n)
        bad = GDN_DEV_ACCEPT_BAD;
    else if (dst < 0 || dst >= a.num_slots)
        bad = GDN_DEV_SLOT_OOR;
    else if (t0 < 0 || int64_t(t0) + j >= a.row_capacity)
        bad = GDN_DEV_ROWS_BAD;
    if (bad) {
        if (c == 0 && threadIdx.x == 0) gdn::set_status(a.status, bad);
        return;
    }
    const int64_t off = int64_t(c) * kChunkFloats;
    const int64_t nf = min(int64_t(kChunkFloats), a.s_elems - off);
    const float4 *src = reinterpret_cast<const float4 *>(a.ckpt + int64_t(l) * a.ckpt_layer_stride +
                                                         (int64_t(t0) + j) * a.s_elems + off);
    float4 *dp = reinterpret_cast<float4 *>(a.pool + int64_t(dst) * a.slot_stride + int64_t(l) * a.layer_stride + off);
    const int n4 = int(nf / 4);
    if (n4 == kChunkFloats / 4) {
        float4 buf[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) buf[u] = __ldcs(src + threadIdx.x + u * kThreads);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) __stcs(dp + threadIdx.x + u * kThreads, buf[u]);
    } else {
        for (int i = threadIdx.x; i < n4; i += kThreads) __stcs(dp + i, __ldcs(src + i));
    }
}

// Zero-copy commit: each (request, layer) location is pointed at its accepted
// checkpoint, under the same tag checks as the copying commit.
struct LocArgs {
    int32_t B, L, row_capacity;
    const int32_t *cu_rows, *accept_len;
    int64_t ckpt_off, ckpt_layer_stride, s_elems;
    const uint64_t *tag;
    uint32_t txn;
    int64_t *loc;
    uint32_t *status;
    int32_t gated;  // as CommitArgs::gated
};

__global__ void __launch_bounds__(kThreads) gdn_commit_at_kernel(const LocArgs a) {
    gdn::pdl_enter();
    const long long idx = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (idx >= (long long)a.B * a.L) return;
    if (a.status && (*reinterpret_cast<volatile uint32_t *>(a.status) & GDN_DEV_TIMEOUT)) return;
    const int r = int(idx % a.B);
    const int l = int(idx / a.B);
    const uint64_t tag = a.tag[int64_t(l) * a.B + r];
    const int j = a.accept_len[r];
    const int t0 = a.cu_rows[r];
    const uint32_t n = uint32_t(tag & 0xffffffffull);
    if (a.gated && j < 0) return;
    uint32_t bad = 0;
    if (uint32_t(tag >> 32) != a.txn || n == 0)
        bad = GDN_DEV_CKPT_UNWRITTEN;
    else if (j < 0 || uint32_t(j) >= n)
        bad = GDN_DEV_ACCEPT_BAD;
    else if (t0 < 0 || int64_t(t0) + j >= a.row_capacity)
        bad = GDN_DEV_ROWS_BAD;
    if (bad) {
        gdn::set_status(a.status, bad);
        return;
    }
    a.loc[int64_t(l) * a.B + r] = a.ckpt_off + int64_t(l) * a.ckpt_layer_stride + (int64_t(t0) + j) * a.s_elems;
}

// Copies every (request, layer) state from its location into the request's slot.
struct MatArgs {
    int32_t B, L, num_slots, chunks;
    const float *base;
    int64_t max_off, s_elems, slot_stride, layer_stride;
    const int64_t *loc;
    float *pool;
    const int32_t *dst_slot;
    uint32_t *status;
};

__global__ void __launch_bounds__(kThreads) gdn_materialize_kernel(const MatArgs a) {
    gdn::pdl_enter();
    const long long idx = blockIdx.x;
    const int c = int(idx % a.chunks);
    const long long rl = idx / a.chunks;
    const int r = int(rl % a.B);
    const int l = int(rl / a.B);
    const int64_t off = a.loc[int64_t(l) * a.B + r];
    const int dst = a.dst_slot[r];
    if (off < 0 || off > a.max_off || (off & 3) != 0 || dst < 0 || dst >= a.num_slots) {
        if (c == 0 && threadIdx.x == 0) gdn::set_status(a.status, GDN_DEV_SLOT_OOR);
        return;
    }
    const float *src = a.base + off;
    float *dp = a.pool + int64_t(dst) * a.slot_stride + int64_t(l) * a.layer_stride;
    if (src == dp) return;  // already in place
    const int64_t o0 = int64_t(c) * kChunkFloats;
    const int n4 = int(min(int64_t(kChunkFloats), a.s_elems - o0) / 4);
    const float4 *s4 = reinterpret_cast<const float4 *>(src + o0);
    float4 *d4 = reinterpret_cast<float4 *>(dp + o0);
    for (int i = threadIdx.x; i < n4; i += kThreads) __stcs(d4 + i, __ldcs(s4 + i));
}


// Transaction gate of the host driver ("Native three-step MTP", Results:
// recovery after abort -- a failed step leaves the slot pool as it was).
// One block checks every (request, layer) pair exactly as the commit does,
// and that no bounded wait has run out (GDN_DEV_TIMEOUT in the status word).
// If anything fails it reports the cause in the status word and sets every
// accept length to -1, so that the gated commit that follows writes nothing
// at all (not even for the pairs that passed) and the host, which reads the
// accept lengths back, undoes the whole transaction.
struct GateArgs {
    int32_t B, L, row_capacity, num_slots;
    const int32_t *cu_rows, *dst_slot;  // dst_slot NULL: zero-copy commit
    int32_t *accept_len;
    const uint64_t *tag;
    uint32_t txn;
    uint32_t *status;
};

constexpr int kGateThreads = 1024;

__global__ void __launch_bounds__(kGateThreads) gdn_commit_gate_kernel(const GateArgs a) {
    __shared__ uint32_t bad_all;
    if (threadIdx.x == 0) bad_all = 0;
    __syncthreads();
    uint32_t bad = 0;
    if (threadIdx.x == 0 && a.status && (*reinterpret_cast<volatile uint32_t *>(a.status) & GDN_DEV_TIMEOUT))
        bad |= GDN_DEV_TIMEOUT;
    const long long pairs = (long long)a.B * a.L;
    for (long long idx = threadIdx.x; idx < pairs; idx += kGateThreads) {
        const int r = int(idx % a.B);
        const int l = int(idx / a.B);
        const uint64_t tag = a.tag[int64_t(l) * a.B + r];
        const int j = a.accept_len[r];
        const int t0 = a.cu_rows[r];
        const uint32_t n = uint32_t(tag & 0xffffffffull);
        if (uint32_t(tag >> 32) != a.txn || n == 0)
            bad |= GDN_DEV_CKPT_UNWRITTEN;
        else if (j < 0 || uint32_t(j) >= n)
            bad |= GDN_DEV_ACCEPT_BAD;
        else if (a.dst_slot && (a.dst_slot[r] < 0 || a.dst_slot[r] >= a.num_slots))
            bad |= GDN_DEV_SLOT_OOR;
        else if (t0 < 0 || int64_t(t0) + j >= a.row_capacity)
            bad |= GDN_DEV_ROWS_BAD;
    }
    if (bad) atomicOr(&bad_all, bad);
    __syncthreads();
    const uint32_t b = bad_all;
    __syncthreads();  // every accept length is read before any is cleared
    if (b == 0) return;
    if (threadIdx.x == 0) gdn::set_status(a.status, b);
    for (int r = threadIdx.x; r < a.B; r += kGateThreads) a.accept_len[r] = -1;
}
}  // namespace

static int commit_at_impl(int gated, const gdn_dims *dims, int32_t B, int32_t num_layers, int32_t row_capacity,
                          const int32_t *cu_rows, const int32_t *accept_len, int64_t ckpt_off,
                          int64_t ckpt_layer_stride, const uint64_t *ckpt_tag, uint32_t txn, int64_t *loc,
                          uint32_t *dev_status, void *stream) {
    if (!dims) return GDN_ERR_NULL;
    if (!gdn_host::dims_ok(dims)) return GDN_ERR_SHAPE;
    if (B < 0 || num_layers < 0 || row_capacity < 0 || ckpt_off < 0) return GDN_ERR_ARG;
    if (B == 0 || num_layers == 0) return GDN_OK;
    if (!cu_rows || !accept_len || !ckpt_tag || !loc) return GDN_ERR_NULL;
    const int64_t se = int64_t(dims->h_v) * dims->d_v * dims->d_k;
    if (ckpt_layer_stride < se * row_capacity || (ckpt_off % 4) != 0 || (ckpt_layer_stride % 4) != 0)
        return GDN_ERR_ARG;
    LocArgs a{};
    a.B = B;
    a.L = num_layers;
    a.row_capacity = row_capacity;
    a.cu_rows = cu_rows;
    a.accept_len = accept_len;
    a.ckpt_off = ckpt_off;
    a.ckpt_layer_stride = ckpt_layer_stride;
    a.s_elems = se;
    a.tag = ckpt_tag;
    a.txn = txn;
    a.loc = loc;
    a.status = dev_status;
    a.gated = gated;
    const long long n = (long long)B * num_layers;
    return gdn_host::launch_pdl(gdn_commit_at_kernel, dim3(unsigned((n + kThreads - 1) / kThreads)), dim3(kThreads), 0,
                                static_cast<cudaStream_t>(stream), a);
}

extern "C" int gdn_materialize(const gdn_dims *dims, int32_t B, int32_t num_layers, const float *state_base,
                               int64_t state_elems_total, const int64_t *loc, float *pool, int64_t slot_stride,
                               int64_t layer_stride, int32_t num_slots, const int32_t *dst_slot,
                               uint32_t *dev_status, void *stream) {
    if (!dims) return GDN_ERR_NULL;
    if (!gdn_host::dims_ok(dims)) return GDN_ERR_SHAPE;
    if (B < 0 || num_layers < 0 || num_slots <= 0) return GDN_ERR_ARG;
    if (B == 0 || num_layers == 0) return GDN_OK;
    if (!state_base || !loc || !pool || !dst_slot) return GDN_ERR_NULL;
    const int64_t se = int64_t(dims->h_v) * dims->d_v * dims->d_k;
    if (state_elems_total < se || layer_stride < se || slot_stride < layer_stride * num_layers) return GDN_ERR_ARG;
    if ((slot_stride | layer_stride) % 4 != 0 || !gdn_host::aligned16(state_base) || !gdn_host::aligned16(pool))
        return GDN_ERR_ARG;
    MatArgs a{};
    a.B = B;
    a.L = num_layers;
    a.num_slots = num_slots;
    a.chunks = int((se + kChunkFloats - 1) / kChunkFloats);
    a.base = state_base;
    a.max_off = state_elems_total - se;
    a.s_elems = se;
    a.slot_stride = slot_stride;
    a.layer_stride = layer_stride;
    a.loc = loc;
    a.pool = pool;
    a.dst_slot = dst_slot;
    a.status = dev_status;
    const long long grid = (long long)B * num_layers * a.chunks;
    if (grid > 0x7fffffffLL) return GDN_ERR_ARG;
    const int st_m = gdn_host::launch_pdl(gdn_materialize_kernel, dim3(unsigned(grid)), dim3(kThreads), 0,
                                          static_cast<cudaStream_t>(stream), a);
    if (st_m != GDN_OK) return st_m;
    return gdn_host::launch_status(cudaGetLastError());
}

static int commit_impl(int gated, const gdn_dims *dims, int32_t B, int32_t num_layers, int32_t row_capacity,
                       const int32_t *cu_rows, const int32_t *accept_len, const float *ckpt,
                       int64_t ckpt_layer_stride, const uint64_t *ckpt_tag, uint32_t txn, float *pool,
                       int64_t slot_stride, int64_t layer_stride, int32_t num_slots, const int32_t *dst_slot,
                       uint32_t *dev_status, void *stream) {
    if (!dims) return GDN_ERR_NULL;
    if (!gdn_host::dims_ok(dims)) return GDN_ERR_SHAPE;
    if (B < 0 || num_layers < 0 || row_capacity < 0 || num_slots <= 0) return GDN_ERR_ARG;
    if (B == 0 || num_layers == 0) return GDN_OK;
    if (!cu_rows || !accept_len || !ckpt || !ckpt_tag || !pool || !dst_slot) return GDN_ERR_NULL;
    const int64_t se = int64_t(dims->h_v) * dims->d_v * dims->d_k;
    if (layer_stride < se || slot_stride < layer_stride * num_layers) return GDN_ERR_ARG;
    if (ckpt_layer_stride < se * row_capacity) return GDN_ERR_ARG;
    if ((slot_stride | layer_stride | ckpt_layer_stride) % 4 != 0) return GDN_ERR_ARG;
    if (!gdn_host::aligned16(ckpt) || !gdn_host::aligned16(pool)) return GDN_ERR_ARG;
    CommitArgs a{};
    a.B = B;
    a.L = num_layers;
    a.row_capacity = row_capacity;
    a.num_slots = num_slots;
    a.chunks = int((se + kChunkFloats - 1) / kChunkFloats);
    a.cu_rows = cu_rows;
    a.accept_len = accept_len;
    a.dst_slot = dst_slot;
    a.ckpt = ckpt;
    a.ckpt_layer_stride = ckpt_layer_stride;
    a.s_elems = se;
    a.slot_stride = slot_stride;
    a.layer_stride = layer_stride;
    a.tag = ckpt_tag;
    a.txn = txn;
    a.pool = pool;
    a.status = dev_status;
    a.gated = gated;
    const long long grid = (long long)B * num_layers * a.chunks;
    if (grid > 0x7fffffffLL) return GDN_ERR_ARG;
    return gdn_host::launch_pdl(gdn_commit_kernel, dim3(unsigned(grid)), dim3(kThreads), 0,
                                static_cast<cudaStream_t>(stream), a);
}

extern "C" int gdn_commit(const gdn_dims *dims, int32_t B, int32_t num_layers, int32_t row_capacity,
                          const int32_t *cu_rows, const int32_t *accept_len, const float *ckpt,
                          int64_t ckpt_layer_stride, const uint64_t *ckpt_tag, uint32_t txn, float *pool,
                          int64_t slot_stride, int64_t layer_stride, int32_t num_slots, const int32_t *dst_slot,
                          uint32_t *dev_status, void *stream) {
    return commit_impl(0, dims, B, num_layers, row_capacity, cu_rows, accept_len, ckpt, ckpt_layer_stride,
                       ckpt_tag, txn, pool, slot_stride, layer_stride, num_slots, dst_slot, dev_status, stream);
}

extern "C" int gdn_commit_at(const gdn_dims *dims, int32_t B, int32_t num_layers, int32_t row_capacity,
                             const int32_t *cu_rows, const int32_t *accept_len, int64_t ckpt_off,
                             int64_t ckpt_layer_stride, const uint64_t *ckpt_tag, uint32_t txn, int64_t *loc,
                             uint32_t *dev_status, void *stream) {
    return commit_at_impl(0, dims, B, num_layers, row_capacity, cu_rows, accept_len, ckpt_off, ckpt_layer_stride,
                          ckpt_tag, txn, loc, dev_status, stream);
}

// The host driver's all-or-nothing commit: the transaction gate, then the
// commit in gated mode (internal to the library; driver.cu).
static int gate_launch(int32_t B, int32_t num_layers, int32_t row_capacity, const int32_t *cu_rows,
                       int32_t *accept_len, const uint64_t *ckpt_tag, uint32_t txn, const int32_t *dst_slot,
                       int32_t num_slots, uint32_t *dev_status, cudaStream_t st) {
    GateArgs g{};
    g.B = B;
    g.L = num_layers;
    g.row_capacity = row_capacity;
    g.num_slots = num_slots;
    g.cu_rows = cu_rows;
    g.dst_slot = dst_slot;
    g.accept_len = accept_len;
    g.tag = ckpt_tag;
    g.txn = txn;
    g.status = dev_status;
    gdn_commit_gate_kernel<<<1, kGateThreads, 0, st>>>(g);
    return gdn_host::launch_status(cudaGetLastError());
}

int gdn_gated_commit(const gdn_dims *dims, int32_t B, int32_t num_layers, int32_t row_capacity,
                     const int32_t *cu_rows, int32_t *accept_len, const float *ckpt, int64_t ckpt_layer_stride,
                     const uint64_t *ckpt_tag, uint32_t txn, float *pool, int64_t slot_stride, int64_t layer_stride,
                     int32_t num_slots, const int32_t *dst_slot, uint32_t *dev_status, void *stream) {
    if (!dims || !cu_rows || !accept_len || !ckpt_tag || !dst_slot) return GDN_ERR_NULL;
    if (B <= 0 || num_layers <= 0) return GDN_ERR_ARG;
    const int st = gate_launch(B, num_layers, row_capacity, cu_rows, accept_len, ckpt_tag, txn, dst_slot, num_slots,
                               dev_status, static_cast<cudaStream_t>(stream));
    if (st != GDN_OK) return st;
    return commit_impl(1, dims, B, num_layers, row_capacity, cu_rows, accept_len, ckpt, ckpt_layer_stride, ckpt_tag,
                       txn, pool, slot_stride, layer_stride, num_slots, dst_slot, dev_status, stream);
}

int gdn_gated_commit_at(const gdn_dims *dims, int32_t B, int32_t num_layers, int32_t row_capacity,
                        const int32_t *cu_rows, int32_t *accept_len, int64_t ckpt_off, int64_t ckpt_layer_stride,
                        const uint64_t *ckpt_tag, uint32_t txn, int64_t *loc, uint32_t *dev_status, void *stream) {
    if (!dims || !cu_rows || !accept_len || !ckpt_tag) return GDN_ERR_NULL;
    if (B <= 0 || num_layers <= 0) return GDN_ERR_ARG;
    const int st = gate_launch(B, num_layers, row_capacity, cu_rows, accept_len, ckpt_tag, txn, nullptr, 0,
                               dev_status, static_cast<cudaStream_t>(stream));
    if (st != GDN_OK) return st;
    return commit_at_impl(1, dims, B, num_layers, row_capacity, cu_rows, accept_len, ckpt_off, ckpt_layer_stride,
                          ckpt_tag, txn, loc, dev_status, stream);
}
