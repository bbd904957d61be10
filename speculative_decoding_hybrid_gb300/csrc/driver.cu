// Host driver of one decode transaction: the plan, the device work of every
// layer and the one device-to-host read, issued by the library in one call.
//
// "Run chained MTP drafting in the batch Engine", Summary: the engine plans
// each transaction (per-request draft lengths), verifies every layer, accepts
// on the device and reads the accepted ids back once at the end; Correctness
// fix: a rejected draft rolls each layer back to its accepted checkpoint.
// "Native three-step MTP", Results: a failed step leaves the slot pool as it
// was (recovery after abort).
//
// The calls made here are the library's own entry points, in the order a
// caller would make them; this file only removes the host glue between them
// (plus one small kernel that moves the step's tables through mapped host
// memory instead of the copy engines).
#include <cuda_runtime.h>
#include <string.h>

#include "gdnspec.h"

// The all-or-nothing commit of a driven transaction (gdn_commit.cu): a gate
// kernel checks every (request, layer) pair first and, if any fails, sets
// every accept length to -1 so that nothing is committed.
int gdn_gated_commit(const gdn_dims *dims, int32_t B, int32_t num_layers, int32_t row_capacity,
                     const int32_t *cu_rows, int32_t *accept_len, const float *ckpt, int64_t ckpt_layer_stride,
                     const uint64_t *ckpt_tag, uint32_t txn, float *pool, int64_t slot_stride, int64_t layer_stride,
                     int32_t num_slots, const int32_t *dst_slot, uint32_t *dev_status, void *stream);
int gdn_gated_commit_at(const gdn_dims *dims, int32_t B, int32_t num_layers, int32_t row_capacity,
                        const int32_t *cu_rows, int32_t *accept_len, int64_t ckpt_off, int64_t ckpt_layer_stride,
                        const uint64_t *ckpt_tag, uint32_t txn, int64_t *loc, uint32_t *dev_status, void *stream);

namespace {

// Six timing events per host thread and device, created on first use.
struct StepEvents {
    int device = -1;
    cudaEvent_t ev[6] = {};
};

bool step_events(StepEvents &se) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (se.device == dev) return true;
    for (auto &e : se.ev)
        if (e) {
            cudaEventDestroy(e);
            e = nullptr;
        }
    se.device = -1;
    for (auto &e : se.ev)
        if (cudaEventCreate(&e) != cudaSuccess) return false;
    se.device = dev;
    return true;
}

thread_local StepEvents t_events;

// Small host <-> device table moves by a kernel over page-locked host memory
// mapped into the device address space, so that they never queue behind a
// large copy the caller has put on a copy engine (the next transaction's
// inputs, say): three spans of n[k] int32 each, copied by one block.
struct Spans {
    const int32_t *src[3];
    int32_t *dst[3];
    int32_t n[3];
};

__global__ void move_spans_kernel(const Spans sp) {
#pragma unroll
    for (int k = 0; k < 3; ++k)
        for (int i = threadIdx.x; i < sp.n[k]; i += blockDim.x) sp.dst[k][i] = sp.src[k][i];
}

// The device address of mapped page-locked host memory, or nullptr.
int32_t *mapped(int32_t *host) {
    void *d = nullptr;
    if (cudaHostGetDevicePointer(&d, host, 0) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return static_cast<int32_t *>(d);
}

// One decode transaction; `arena` selects the zero-copy form (start states
// at arena locations, checkpoints in the area of the transaction's parity,
// commit by rewriting locations) instead of the slot-pool form.
int run_transaction(const gdn_dims *dims, int32_t num_layers, int32_t row_capacity, gdn_req *reqs, int32_t n_reqs,
                    const gdn_plan_limits *lim, gdn_pool *pool, gdn_plan *plan, uint32_t *txn,
                    const gdn_decode_io *io, const gdn_arena_io *arena, float *kernel_ms, void *stream) {
    if (!dims || !reqs || !lim || !pool || !plan || !txn || !io) return GDN_ERR_NULL;
    if (!io->tables || !io->rows || !io->host_tables || !io->host_out || !io->accept_len || !io->bonus ||
        !io->out_tokens)
        return GDN_ERR_NULL;
    if (arena && (!arena->arena || !arena->loc)) return GDN_ERR_NULL;
    if (n_reqs <= 0 || num_layers <= 0 || row_capacity <= 0) return GDN_ERR_ARG;
    for (int32_t i = 0; i < n_reqs; ++i)
        if (reqs[i].kind != GDN_REQ_DECODE) return GDN_ERR_ARG;  // decode transactions only; nothing planned
    int st = plan_transaction(reqs, n_reqs, lim, pool, plan);
    if (st != GDN_OK) return st;
    const int32_t B = plan->n_decode;
    const int32_t rows = plan->decode_rows;
    // The location table is laid out per request: every request must be in the transaction.
    if (plan->n_prefill > 0 || B <= 0 || rows > row_capacity || (arena && B != n_reqs)) {
        gdn_pool_abort(pool, plan, n_reqs);
        return GDN_ERR_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int32_t W = n_reqs + 1;
    int32_t *h = io->host_tables;
    memcpy(h, plan->dec_cu, size_t(B + 1) * 4);
    memcpy(h + W, plan->dec_src, size_t(B) * 4);
    memcpy(h + 2 * W, plan->dec_dst, size_t(B) * 4);
    const int32_t *cu = io->tables;
    const int32_t *src = io->tables + W;
    const int32_t *dst = io->tables + 2 * W;
    bool timing = kernel_ms != nullptr && step_events(t_events);
    cudaEvent_t *ev = t_events.ev;
    const uint32_t t = *txn + 1u;
    const int64_t area = arena ? arena->area_off[t & 1u] : 0;
    auto fail = [&](int code) {
        gdn_pool_abort(pool, plan, n_reqs);
        return code;
    };
    int32_t *h_dev = mapped(h);
    if (h_dev) {
        Spans sp{{h_dev, h_dev + W, h_dev + 2 * W}, {io->tables, io->tables + W, io->tables + 2 * W}, {B + 1, B, B}};
        move_spans_kernel<<<1, 256, 0, s>>>(sp);
        if (cudaGetLastError() != cudaSuccess) return fail(GDN_ERR_CUDA);
    } else if (cudaMemcpyAsync(io->tables, h, size_t(3) * W * 4, cudaMemcpyHostToDevice, s) != cudaSuccess) {
        return fail(GDN_ERR_CUDA);
    }
    if (timing) cudaEventRecord(ev[0], s);
    if (arena)
        st = gdn_verify_at_layers(dims, num_layers, B, row_capacity, cu, io->rows, arena->arena, arena->elems_total,
                                  arena->loc, arena->arena + area, io->ckpt_layer_stride, io->ckpt_tag, t, io->o,
                                  io->o_layer_stride, io->dev_status, stream);
    else
        st = gdn_verify_layers(dims, num_layers, B, row_capacity, cu, io->rows, io->pool, io->slot_stride,
                               io->layer_stride, io->num_slots, src, io->ckpt, io->ckpt_layer_stride, io->ckpt_tag,
                               t, io->o, io->o_layer_stride, io->dev_status, stream);
    if (st != GDN_OK) return fail(st);
    if (timing) {
        cudaEventRecord(ev[1], s);
        cudaEventRecord(ev[2], s);
    }
    st = mtp_greedy_accept(B, row_capacity, cu, io->logits, io->vocab, io->logit_row_stride, io->tokens, io->argmax,
                           io->accept_len, io->bonus, io->out_tokens, io->stats, io->workspace, io->workspace_bytes,
                           io->dev_status, stream);
    if (st != GDN_OK) return fail(st);
    if (timing) {
        cudaEventRecord(ev[3], s);
        cudaEventRecord(ev[4], s);
    }
    // All or nothing: a device-detected problem anywhere in the transaction
    // (a stale or missing checkpoint, a bad accept length or slot, a wait
    // that ran out) commits no pair at all and marks every accept length -1.
    if (arena)
        st = gdn_gated_commit_at(dims, B, num_layers, row_capacity, cu, io->accept_len, area,
                                 io->ckpt_layer_stride, io->ckpt_tag, t, arena->loc, io->dev_status, stream);
    else
        st = gdn_gated_commit(dims, B, num_layers, row_capacity, cu, io->accept_len, io->ckpt,
                              io->ckpt_layer_stride, io->ckpt_tag, t, io->pool, io->slot_stride, io->layer_stride,
                              io->num_slots, dst, io->dev_status, stream);
    if (st != GDN_OK) return fail(st);
    if (timing) cudaEventRecord(ev[5], s);
    int32_t *ho = io->host_out;
    int32_t *ho_dev = mapped(ho);
    bool moved = false;
    if (ho_dev) {
        Spans sp{{io->accept_len, io->bonus, io->out_tokens}, {ho_dev, ho_dev + n_reqs, ho_dev + 2 * n_reqs},
                 {B, B, rows}};
        move_spans_kernel<<<1, 256, 0, s>>>(sp);
        moved = cudaGetLastError() == cudaSuccess;
    } else {
        moved = cudaMemcpyAsync(ho, io->accept_len, size_t(B) * 4, cudaMemcpyDeviceToHost, s) == cudaSuccess &&
                cudaMemcpyAsync(ho + n_reqs, io->bonus, size_t(B) * 4, cudaMemcpyDeviceToHost, s) == cudaSuccess &&
                cudaMemcpyAsync(ho + 2 * n_reqs, io->out_tokens, size_t(rows) * 4, cudaMemcpyDeviceToHost, s) ==
                    cudaSuccess;
    }
    if (!moved || cudaStreamSynchronize(s) != cudaSuccess) return fail(GDN_ERR_CUDA);
    if (timing) {
        for (int i = 0; i < 3; ++i)
            if (cudaEventElapsedTime(&kernel_ms[i], ev[2 * i], ev[2 * i + 1]) != cudaSuccess) kernel_ms[i] = -1.f;
    }
    // A refused transaction committed nothing: its fresh slots return to the
    // pool and the requests, the pool and the transaction counter stay as
    // they were (in the zero-copy form the next transaction then writes the
    // same checkpoint area again, never the one the locations point into).
    for (int32_t j = 0; j < B; ++j)
        if (ho[j] < 0) return fail(GDN_ERR_REFUSED);
    *txn = t;
    // The commit is done: requests that moved release their old slot, and
    // every decode request advances by its accepted drafts plus the bonus.
    st = gdn_pool_apply(pool, plan, n_reqs);
    if (st != GDN_OK) return st;
    for (int32_t j = 0; j < B; ++j) {
        const int32_t i = plan->dec_req[j];
        reqs[i].slot = plan->dst[i];
        reqs[i].cur_len += ho[j] + 1;
    }
    return GDN_OK;
}

}  // namespace

extern "C" int gdn_decode_transaction(const gdn_dims *dims, int32_t num_layers, int32_t row_capacity,
                                      gdn_req *reqs, int32_t n_reqs, const gdn_plan_limits *lim, gdn_pool *pool,
                                      gdn_plan *plan, uint32_t *txn, const gdn_decode_io *io, float *kernel_ms,
                                      void *stream) {
    return run_transaction(dims, num_layers, row_capacity, reqs, n_reqs, lim, pool, plan, txn, io, nullptr,
                           kernel_ms, stream);
}

extern "C" int gdn_decode_transaction_at(const gdn_dims *dims, int32_t num_layers, int32_t row_capacity,
                                         gdn_req *reqs, int32_t n_reqs, const gdn_plan_limits *lim, gdn_pool *pool,
                                         gdn_plan *plan, uint32_t *txn, const gdn_decode_io *io,
                                         const gdn_arena_io *arena, float *kernel_ms, void *stream) {
    if (!arena) return GDN_ERR_NULL;
    return run_transaction(dims, num_layers, row_capacity, reqs, n_reqs, lim, pool, plan, txn, io, arena, kernel_ms,
                           stream);
}
