/*
 * gdnspec -- K-draft MTP speculative verification over GatedDeltaNet layers,
 * for one GB300 (sm_103a).  C ABI.
 *
 * Sources the operations follow (page title, section):
 *   [NATIVE]  "Native three-step MTP": What changed (FP32 sigmoid gates; GDN
 *             state-update rounding identical in decode and verification;
 *             prefill state published before dependent decode/verify),
 *             Results (shared-prefix protection, duplicate-slot release,
 *             rejected requests, recovery after abort).
 *   [ENGINE]  "Run chained MTP drafting in the batch Engine": Summary
 *             (per-request draft lengths, device-resident draft ids with one
 *             final host read, C-visible telemetry, draft deferral for
 *             transactions mixing prefill and speculative rows), Correctness
 *             fix (chunked GatedDeltaNet publishes only the final state, not
 *             the per-row recurrent checkpoints needed to reject drafts),
 *             H200 RC4 evidence (mixed K, rollback, max-length clamping).
 *   [CARD]    "Accio-Lab/occamy-1.0-MTP": MTP1 runtime (unsupported
 *             batch shapes fail closed).
 *
 * The recurrence (gated delta rule), per v-head h with qk-head h / (h_v/h_qk):
 *     S_t = S_{t-1} alpha_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *     o_t = q_scale * S_t q_t,    alpha_t = expf(g_t)  (FP32).
 * g_t is the log-decay and beta_t the write strength; both are FP32 values
 * already passed through the model's sigmoid (kept in FP32, [NATIVE]).
 *
 * Conventions shared by every entry point
 *   - Tensor pointers are DEVICE pointers unless a parameter says "host".
 *     The caller owns every buffer; the library allocates no device memory.
 *     Its only global state is the fixed scratch array of
 *     mtp_greedy_accept_noalloc (see there).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Errors that the host can see (null pointers, shapes,
 *     sizes) are returned at once and nothing is launched.  Errors only the
 *     device can see (slot or row tables, token ids, stale checkpoints) set
 *     bits in *dev_status (atomicOr) and skip the offending request; other
 *     requests proceed.  No kernel traps, asserts or waits without a bound.
 *   - dev_status accumulates until the caller clears it.
 *   - Layouts (row-major, innermost last):
 *       q, k   bf16 [rows][h_qk][d_k]       v, o   bf16 [rows][h_v][d_v]
 *       g,beta fp32 [rows][h_v]
 *       state  fp32 [h_v][d_v][d_k]  (S[a][j]: a over values, j over keys)
 *       pool   slot s, layer l at  pool + s*slot_stride + l*layer_stride
 *       ckpt   fp32 [rows][h_v][d_v][d_k] per layer (packed row index)
 *     Packed rows: request r owns rows cu_rows[r] .. cu_rows[r+1]-1; row 0 of
 *     a request is its last committed token, rows 1..K its drafts.
 *   - Supported shapes: d_k = d_v in {16, 32, 64, 128}; h_v a multiple of
 *     h_qk; rows per request 1 .. GDN_MAX_ROWS.  Anything else returns
 *     GDN_ERR_SHAPE (fail closed, [CARD]).
 */
#ifndef GDNSPEC_H
#define GDNSPEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t gdn_bf16;          /* bf16 bit pattern */

#define GDN_K_MAX 15                /* drafts per request */
#define GDN_MAX_ROWS (GDN_K_MAX + 1)

/* Return codes */
enum {
    GDN_OK = 0,
    GDN_ERR_NULL = -1,       /* a required pointer is NULL */
    GDN_ERR_SHAPE = -2,      /* unsupported head sizes / grouping */
    GDN_ERR_ARG = -3,        /* bad size, stride, count or slot */
    GDN_ERR_DUP_SLOT = -4,   /* two requests would write one slot */
    GDN_ERR_NO_SLOT = -5,    /* free list empty */
    GDN_ERR_CUDA = -6,       /* a CUDA launch or query failed */
    GDN_ERR_WORKSPACE = -7,  /* workspace missing or too small */
    GDN_ERR_REFUSED = -8     /* a device-side check refused a driven transaction; nothing committed */
};

/* Bits of *dev_status */
enum {
    GDN_DEV_SLOT_OOR = 1u,        /* slot id outside [0, num_slots) */
    GDN_DEV_ROWS_BAD = 2u,        /* cu_rows not monotone, rows outside 1..GDN_MAX_ROWS or past capacity */
    GDN_DEV_TOKEN_OOR = 4u,       /* draft id outside [0, vocab): counted as a miss */
    GDN_DEV_CKPT_UNWRITTEN = 8u,  /* commit asked for a checkpoint not written in this transaction */
    GDN_DEV_ACCEPT_BAD = 16u,     /* accept length outside [0, rows written) */
    GDN_DEV_TIMEOUT = 32u         /* a bounded wait on an asynchronous copy ran out */
};

typedef struct gdn_dims {
    int32_t h_qk, h_v, d_k, d_v;
    float q_scale;                /* multiplies o; 1.0 for the plain rule */
} gdn_dims;

/* Cumulative speculative telemetry ([ENGINE] Summary), device-resident. */
typedef struct mtp_stats {
    uint64_t proposed;    /* drafts offered                        */
    uint64_t evaluated;   /* drafts compared, up to the first miss */
    uint64_t accepted;    /* drafts accepted                       */
    uint64_t emitted;     /* tokens emitted (accepted + bonus)     */
    uint64_t steps;       /* accept calls                          */
} mtp_stats;

/*
 * gdn_decode_step -- one token per request ([NATIVE] What changed; [ENGINE]
 * Correctness fix: decode requests advance by one token).
 *   B requests; row r of q,k,v,g,beta,o belongs to request r.
 *   Reads the state of slot src_slot[r] of this layer, writes the advanced
 *   state to dst_slot[r] (in place when equal) and o[r].
 *   pool_layer = pool + l*layer_stride; slot stride in floats.
 * The per-token arithmetic is the same code, in the same order, as
 * gdn_verify's: a verify checkpoint j is bit-identical to j+1 decode steps.
 * Distinct requests must not name the same dst_slot, and no request's
 * dst_slot may be another request's src_slot (plan_transaction guarantees it).
 */
int gdn_decode_step(const gdn_dims *dims, int32_t B,
                    const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                    const float *g, const float *beta,
                    float *pool_layer, int64_t slot_stride, int32_t num_slots,
                    const int32_t *src_slot, const int32_t *dst_slot,
                    gdn_bf16 *o, uint32_t *dev_status, void *stream);

/*
 * gdn_verify -- fused K-draft verification of one layer ([ENGINE]
 * Correctness fix: the intermediate recurrent checkpoints required to reject
 * drafts; Summary: per-request draft lengths).
 *   For request r (rows cu_rows[r] .. cu_rows[r+1]-1, 1..GDN_MAX_ROWS of
 *   them) the state of slot src_slot[r] is advanced row by row; after row t
 *   the state is written to ckpt_layer[t] and o[t] = bf16(q_scale * S_t q_t).
 *   The slot itself is never written (the step is a transaction until
 *   gdn_commit).  row_capacity bounds every row-indexed buffer (q,k,v,g,
 *   beta,o,ckpt_layer): requests reaching past it are refused (ROWS_BAD).
 *   ckpt_tag[r] (this layer's tag array) receives (txn << 32) | rows, or
 *   (txn << 32) | 0 when the request was refused; gdn_commit only copies a
 *   checkpoint whose tag carries the same txn.
 */
int gdn_verify(const gdn_dims *dims, int32_t B, int32_t row_capacity,
               const int32_t *cu_rows,
               const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
               const float *g, const float *beta,
               const float *pool_layer, int64_t slot_stride, int32_t num_slots,
               const int32_t *src_slot,
               float *ckpt_layer, uint64_t *ckpt_tag, uint32_t txn,
               gdn_bf16 *o, uint32_t *dev_status, void *stream);

/* Per-layer row inputs for the multi-layer calls below (device pointers). */
typedef struct gdn_layer_rows {
    const gdn_bf16 *q, *k, *v;
    const float *g, *beta;
} gdn_layer_rows;

/*
 * gdn_verify_layers -- num_layers gdn_verify calls issued from the library in
 *   layer order on `stream` (the same kernels, arguments and results as
 *   calling gdn_verify per layer): layer l reads rows[l] (host array of
 *   device pointers), the slots at pool + l*layer_stride, writes checkpoints
 *   at ckpt + l*ckpt_layer_stride, tags at ckpt_tag + l*B and outputs at
 *   o + l*o_layer_stride.  For callers that hold every layer's inputs (a
 *   multi-layer verifier, a benchmark): it removes the per-layer host call.
 *   Stops at the first layer whose call fails and returns that status.
 */
int gdn_verify_layers(const gdn_dims *dims, int32_t num_layers, int32_t B, int32_t row_capacity,
                      const int32_t *cu_rows, const gdn_layer_rows *rows,
                      const float *pool, int64_t slot_stride, int64_t layer_stride,
                      int32_t num_slots, const int32_t *src_slot,
                      float *ckpt, int64_t ckpt_layer_stride, uint64_t *ckpt_tag, uint32_t txn,
                      gdn_bf16 *o, int64_t o_layer_stride, uint32_t *dev_status, void *stream);

/*
 * mtp_greedy_accept -- greedy acceptance ([NATIVE] greedy requests; [ENGINE]
 * Quality follow-up: verification-row selection and per-request bonus;
 * Summary: device-resident ids, telemetry).
 *   argmax[t] = first index of the largest logit of row t (bf16 compared
 *   exactly; the first NaN wins).  For request r with K = rows-1 drafts:
 *   accept_len[r] = j = number of leading drafts i (1..K) with
 *   tokens[t0+i] == argmax[t0+i-1]; bonus[r] = argmax[t0+j];
 *   out_tokens[t0+m] = argmax[t0+m] for m <= j (the emitted tokens), -1 after.
 *   stats (if not NULL) += {K, min(j+1,K), j, j+1}; steps += 1 per call.
 *   logits: bf16 [row_capacity][row_stride], vocab <= row_stride elements used.
 *   workspace: device scratch of mtp_accept_workspace_bytes(row_capacity, vocab)
 *   bytes (partial maxima of row splits); contents need no initialisation.
 *   A request with bad rows gets accept_len = bonus = -1 (ROWS_BAD).
 */
size_t mtp_accept_workspace_bytes(int32_t row_capacity, int64_t vocab);
int mtp_greedy_accept(int32_t B, int32_t row_capacity, const int32_t *cu_rows,
                      const gdn_bf16 *logits, int64_t vocab, int64_t row_stride,
                      const int32_t *tokens, int32_t *argmax, int32_t *accept_len,
                      int32_t *bonus, int32_t *out_tokens, mtp_stats *stats,
                      void *workspace, size_t workspace_bytes,
                      uint32_t *dev_status, void *stream);

/*
 * mtp_greedy_accept_noalloc -- mtp_greedy_accept without a workspace, for
 * callers that cannot allocate device memory (a plugin whose host engine owns
 * all device memory, or a latency-critical loop that cannot afford a
 * cudaMalloc).  The pages describe no such call; it computes exactly what
 * mtp_greedy_accept computes, with the same arguments minus the workspace.
 *   Scratch: a fixed 512 KiB device array inside the library (held by every
 *   device that loads it until exit), shared by all calls and keeping the
 *   last call's contents.  A request whose mtp_accept_workspace_bytes()
 *   exceeds 512 KiB returns GDN_ERR_WORKSPACE and launches nothing.  Calls
 *   that overlap on the GPU race on the scratch: order them on one stream.
 *   The first call on a device resolves the array's address with that device
 *   current (make it before any stream capture); the stream must belong to
 *   the current device.  No call allocates or frees memory.  The resolved
 *   address is kept for the life of the process: after a cudaDeviceReset
 *   of that device it is stale, so do not call this entry point there again.
 */
int mtp_greedy_accept_noalloc(int32_t B, int32_t row_capacity, const int32_t *cu_rows,
                              const gdn_bf16 *logits, int64_t vocab, int64_t row_stride,
                              const int32_t *tokens, int32_t *argmax, int32_t *accept_len,
                              int32_t *bonus, int32_t *out_tokens, mtp_stats *stats,
                              uint32_t *dev_status, void *stream);

/*
 * gdn_commit -- rollback/commit of all layers in one launch ([ENGINE]
 * Correctness fix; RC4 evidence: rollback).  For request r and layer l:
 *   if ckpt_tag[l*B + r] == (txn << 32) | n with 0 <= accept_len[r] < n and
 *   0 <= dst_slot[r] < num_slots, the checkpoint of packed row
 *   cu_rows[r] + accept_len[r] of layer l (ckpt + l*ckpt_layer_stride) is
 *   copied bit for bit to pool + dst_slot[r]*slot_stride + l*layer_stride.
 *   Otherwise nothing is written for (r, l) and CKPT_UNWRITTEN / ACCEPT_BAD /
 *   SLOT_OOR is set.  If *dev_status already holds GDN_DEV_TIMEOUT when the
 *   commit runs, nothing is committed.
 */
int gdn_commit(const gdn_dims *dims, int32_t B, int32_t num_layers,
               int32_t row_capacity, const int32_t *cu_rows,
               const int32_t *accept_len,
               const float *ckpt, int64_t ckpt_layer_stride,
               const uint64_t *ckpt_tag, uint32_t txn,
               float *pool, int64_t slot_stride, int64_t layer_stride,
               int32_t num_slots, const int32_t *dst_slot,
               uint32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Zero-copy commit (the slot table points at the accepted checkpoint).
 * A "state arena" is one fp32 buffer holding the pool slots and two
 * checkpoint areas used on alternate transactions; the state of (request r,
 * layer l) lives at state_base + loc[l*B + r] (element offset).  Instead of
 * copying 2*S_bytes per (request, layer) the commit rewrites loc; the next
 * transaction verifies from there while writing its checkpoints into the
 * other area ([ENGINE] Correctness fix: rollback to the accepted checkpoint;
 * H200 RC4 evidence: the paged Engine addresses state through a table).
 * ------------------------------------------------------------------------ */

/*
 * gdn_verify_at -- gdn_verify whose start states are read at
 *   state_base + src_off[r] (device int64, element offsets, multiples of 4,
 *   each state fully inside [0, state_elems_total)); everything else as in
 *   gdn_verify.  An offset out of range sets GDN_DEV_SLOT_OOR and skips r.
 */
int gdn_verify_at(const gdn_dims *dims, int32_t B, int32_t row_capacity,
                  const int32_t *cu_rows,
                  const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                  const float *g, const float *beta,
                  const float *state_base, int64_t state_elems_total,
                  const int64_t *src_off,
                  float *ckpt_layer, uint64_t *ckpt_tag, uint32_t txn,
                  gdn_bf16 *o, uint32_t *dev_status, void *stream);

/*
 * gdn_commit_at -- for every (request r, layer l) whose checkpoint tag passes
 *   the checks of gdn_commit, set loc[l*B + r] = ckpt_off +
 *   l*ckpt_layer_stride + (cu_rows[r] + accept_len[r]) * S_elems, the element
 *   offset (from the same state_base) of the accepted checkpoint.  Refused
 *   pairs keep their location.  No state bytes move.
 */
int gdn_commit_at(const gdn_dims *dims, int32_t B, int32_t num_layers,
                  int32_t row_capacity, const int32_t *cu_rows,
                  const int32_t *accept_len,
                  int64_t ckpt_off, int64_t ckpt_layer_stride,
                  const uint64_t *ckpt_tag, uint32_t txn,
                  int64_t *loc, uint32_t *dev_status, void *stream);

/*
 * gdn_materialize -- copy the state at state_base + loc[l*B + r] into
 *   pool + dst_slot[r]*slot_stride + l*layer_stride for every (r, l) (a
 *   request leaving the batch, or whose checkpoint area is about to be
 *   reused).  Pairs already in place are skipped; a location out of range or
 *   a bad slot sets GDN_DEV_SLOT_OOR.  Sources and destinations must not
 *   overlap other than being equal.
 */
int gdn_materialize(const gdn_dims *dims, int32_t B, int32_t num_layers,
                    const float *state_base, int64_t state_elems_total,
                    const int64_t *loc, float *pool, int64_t slot_stride,
                    int64_t layer_stride, int32_t num_slots,
                    const int32_t *dst_slot, uint32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Compact fixed-state replay ([ENGINE] closing comment: the runtime rebuilt
 * on compact fixed-state replay without dense recurrent checkpoints).
 * ------------------------------------------------------------------------ */

/*
 * gdn_verify_replay -- verification without checkpoints.  For request r:
 *  1. the previous transaction's accepted rows, prev_cu_rows[r] ..
 *     prev_cu_rows[r] + prev_accept_len[r] (none when prev_accept_len[r] < 0),
 *     are run from slot src_slot[r] through the state update of
 *     gdn_decode_step, and the result is written to slot dst_slot[r] (also
 *     when nothing is pending but dst_slot[r] != src_slot[r]).  This is the
 *     commit of the previous transaction, bit-identical to gdn_commit of its
 *     accepted checkpoint;
 *  2. this transaction's rows cu_rows[r] .. cu_rows[r+1]-1 (0..GDN_MAX_ROWS;
 *     0 rows only commits) run from that state and write o; no state is kept.
 *   prev_k, prev_v (bf16) and prev_g, prev_beta (fp32) are the previous
 *   transaction's rows in the packed layout of gdn_verify (prev_capacity
 *   rows; q is not needed).  Per (request, layer) this moves S_bytes in and
 *   at most S_bytes out instead of (K+2) S_bytes in and (K+2) out.
 *   Rows past either capacity or more accepted rows than existed set
 *   GDN_DEV_ROWS_BAD and skip the request.
 */
int gdn_verify_replay(const gdn_dims *dims, int32_t B, int32_t row_capacity,
                      const int32_t *cu_rows,
                      const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                      const float *g, const float *beta,
                      int32_t prev_capacity, const int32_t *prev_cu_rows,
                      const int32_t *prev_accept_len,
                      const gdn_bf16 *prev_k, const gdn_bf16 *prev_v,
                      const float *prev_g, const float *prev_beta,
                      float *pool_layer, int64_t slot_stride, int32_t num_slots,
                      const int32_t *src_slot, const int32_t *dst_slot,
                      gdn_bf16 *o, uint32_t *dev_status, void *stream);

/*
 * gdn_verify_at_layers -- num_layers gdn_verify_at calls in layer order:
 *   layer l reads rows[l], the start-state offsets src_off + l*B (a [layer]
 *   [request] table), writes checkpoints at ckpt + l*ckpt_layer_stride,
 *   tags at ckpt_tag + l*B and outputs at o + l*o_layer_stride.  Same
 *   contract as the per-layer call; stops at the first failing layer.
 */
int gdn_verify_at_layers(const gdn_dims *dims, int32_t num_layers, int32_t B, int32_t row_capacity,
                         const int32_t *cu_rows, const gdn_layer_rows *rows,
                         const float *state_base, int64_t state_elems_total, const int64_t *src_off,
                         float *ckpt, int64_t ckpt_layer_stride, uint64_t *ckpt_tag, uint32_t txn,
                         gdn_bf16 *o, int64_t o_layer_stride, uint32_t *dev_status, void *stream);

/*
 * gdn_verify_replay_layers -- num_layers gdn_verify_replay calls in layer
 *   order (rows[l] and prev_rows[l] per layer, slots at pool + l*layer_stride,
 *   outputs at o + l*o_layer_stride); same contract as the per-layer call.
 */
int gdn_verify_replay_layers(const gdn_dims *dims, int32_t num_layers, int32_t B, int32_t row_capacity,
                             const int32_t *cu_rows, const gdn_layer_rows *rows,
                             int32_t prev_capacity, const int32_t *prev_cu_rows,
                             const int32_t *prev_accept_len, const gdn_layer_rows *prev_rows,
                             float *pool, int64_t slot_stride, int64_t layer_stride, int32_t num_slots,
                             const int32_t *src_slot, const int32_t *dst_slot,
                             gdn_bf16 *o, int64_t o_layer_stride, uint32_t *dev_status, void *stream);

/*
 * gdn_chunked_prefill -- chunked (WY/UT) GatedDeltaNet prefill of one layer
 * ([ENGINE] Correctness fix: the chunked plan publishes the final state but
 * no per-row checkpoints).  nseq ragged sequences, rows cu_seqlens[i] ..
 * cu_seqlens[i+1]-1 (packed like q,k,v,g,beta,o).  Sequence i starts from
 * slot src_slot[i] (or from zero when src_slot[i] == -1), writes o for every
 * token and publishes only its final state to dst_slot[i].  chunk = 64.
 * dst_slot[i] may equal src_slot[i] (in place); otherwise the destination
 * slots of one call must be distinct and none may be another sequence's
 * source in the same call (sequences run concurrently, so such a read would
 * race with the write; plan_transaction's destinations satisfy this).
 * Work is ordered on `stream`, so a decode/verify queued after it on the
 * same stream reads the published state ([NATIVE] What changed).
 * max_seqlen (host, >= 0) is accepted for callers that track it; every
 * length is read from cu_seqlens on the device.  d_k = d_v = 128 runs on the
 * tensor cores (one CTA per sequence and v-head keeps the state on chip for
 * the whole sequence; nothing but the final state and o is written); 16, 32
 * and 64 run the same chunk form in fp32 on the CUDA cores.
 * Workspace (gdn_prefill_workspace_bytes): the sequences' length order,
 * nseq int32 (16-byte aligned).
 * A sequence whose bounded wait ran out (GDN_DEV_TIMEOUT), and every sequence
 * of a call made while *dev_status already holds GDN_DEV_TIMEOUT, publishes
 * nothing: its destination slot keeps its bytes ([ENGINE] Correctness fix:
 * never publish a state that was not computed in full).
 */
size_t gdn_prefill_workspace_bytes(const gdn_dims *dims, int32_t nseq, int32_t row_capacity);
int gdn_chunked_prefill(const gdn_dims *dims, int32_t nseq, int32_t row_capacity,
                        const int32_t *cu_seqlens, int32_t max_seqlen,
                        const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                        const float *g, const float *beta,
                        float *pool_layer, int64_t slot_stride, int32_t num_slots,
                        const int32_t *src_slot, const int32_t *dst_slot,
                        gdn_bf16 *o, int32_t chunk,
                        void *workspace, size_t workspace_bytes,
                        uint32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Host-side transaction planner and slot pool (HOST memory, synchronous).
 * ------------------------------------------------------------------------ */

enum { GDN_REQ_DECODE = 0, GDN_REQ_PREFILL = 1 };
enum { GDN_PLAN_RECURRENT = 0, GDN_PLAN_CHUNKED = 1 };

typedef struct gdn_req {
    int32_t kind;       /* GDN_REQ_DECODE or GDN_REQ_PREFILL */
    int32_t k_draft;    /* drafts asked for (decode) */
    int32_t n_tokens;   /* prompt tokens still to run (prefill) */
    int32_t cur_len;    /* tokens already in the sequence */
    int32_t max_len;    /* sequence length limit */
    int32_t slot;       /* state slot held, -1 = none (new prefill) */
} gdn_req;

typedef struct gdn_plan_limits {
    int32_t max_rows;   /* row budget of one transaction */
    int32_t max_reqs;   /* request budget of one transaction */
    int32_t k_max;      /* 0 .. GDN_K_MAX */
} gdn_plan_limits;

/* Reference-counted slots; the free list is a FIFO ring.  All storage is
 * caller-owned host memory of num_slots int32 each. */
typedef struct gdn_pool {
    int32_t num_slots;
    int32_t *refcount;
    int32_t *free_fifo;
    int32_t free_head;
    int32_t free_count;
} gdn_pool;

/* free_order (host, may be NULL = 0..num_slots-1) gives the FIFO order. */
int gdn_pool_init(gdn_pool *pool, int32_t num_slots, int32_t *refcount,
                  int32_t *free_fifo, const int32_t *free_order);
int gdn_pool_alloc(gdn_pool *pool, int32_t *slot);       /* GDN_ERR_NO_SLOT when empty */
int gdn_pool_share(gdn_pool *pool, int32_t slot);        /* +1 reference on a held slot */
int gdn_pool_release(gdn_pool *pool, int32_t slot);      /* -1; a free slot -> GDN_ERR_ARG */

/* Plan output.  Scalars are written by plan_transaction; the arrays are
 * caller-owned host buffers of n entries (n+1 for dec_cu and pre_cu). */
typedef struct gdn_plan {
    int32_t n_selected, plan, deferred;
    int32_t n_decode, decode_rows, n_prefill, prefill_rows;
    int32_t *k, *rows, *src, *dst;                 /* per request; k = -1: not selected */
    int32_t *dec_req, *dec_cu, *dec_src, *dec_dst; /* decode group, request order */
    int32_t *pre_req, *pre_cu, *pre_src, *pre_dst; /* prefill group, request order */
} gdn_plan;

/*
 * plan_transaction -- one transaction ([ENGINE] Correctness fix and Summary;
 * RC4 evidence: mixed K, max-length clamping, cache reuse; [NATIVE] Results).
 *  1. Paged selection in request order while rows remain in max_rows and
 *     fewer than max_reqs are taken.  Decode: 1+K rows with
 *     K = max(0, min(k_draft, k_max, max_len-cur_len-1, budget-1)).
 *     Prefill: min(n_tokens, max_len-cur_len, budget) rows.
 *  2. If the selected set holds a prefill and a decode with K > 0, every
 *     selected decode gets K = 0; `deferred` counts the drafts cleared.
 *  3. plan = GDN_PLAN_CHUNKED if a prefill is selected.
 *  4. Slots: a held slot with one reference is written in place; a shared
 *     slot (count > 1) or a new prefill gets a fresh slot (copy-on-write).
 * Errors leave the pool unchanged: GDN_ERR_ARG (bad limits, decode at
 * max_len, empty prefill, slot not held), GDN_ERR_DUP_SLOT, GDN_ERR_NO_SLOT.
 */
int plan_transaction(const gdn_req *reqs, int32_t n, const gdn_plan_limits *lim,
                     gdn_pool *pool, gdn_plan *out);

/* After a successful commit: requests that moved release their old slot. */
int gdn_pool_apply(gdn_pool *pool, const gdn_plan *plan, int32_t n);
/* Abort ([NATIVE] recovery after abort): fresh slots of the plan return to the pool. */
int gdn_pool_abort(gdn_pool *pool, const gdn_plan *plan, int32_t n);

/*
 * gdn_decode_transaction -- one decode transaction in one host call
 * ([ENGINE] Summary: the engine plans, verifies every layer, accepts on the
 * device and reads the results back once; Correctness fix: each layer rolls
 * back to its accepted checkpoint; [NATIVE] Results: recovery after abort).
 * It runs, in order: plan_transaction over reqs; the decode group's tables
 * (cu_rows, src_slot, dst_slot) from io->host_tables (page-locked host,
 * [3][n_reqs+1]) to io->tables (device, same shape) on `stream`;
 * gdn_verify_layers with txn + 1; mtp_greedy_accept; gdn_commit; one
 * device-to-host read into io->host_out (page-locked host, 2*n_reqs +
 * row_capacity int32: accept_len[0..B), bonus at n_reqs.., emitted tokens at
 * 2*n_reqs..); a wait for `stream`; gdn_pool_apply; then for every decoded
 * request i: reqs[i].slot = its destination slot and reqs[i].cur_len +=
 * accept_len + 1.  *txn is the transaction counter (incremented).
 * The commit is all or nothing: before it, one small kernel checks every
 * (request, layer) pair as gdn_commit would (checkpoint tag of this
 * transaction, accept length, destination slot, rows) and that no bounded
 * wait ran out (GDN_DEV_TIMEOUT, which stays set until the caller clears
 * *dev_status: results computed after it are not trusted).  If any check
 * fails, the cause is set in *dev_status, every accept_len becomes -1, no
 * state is written, and the call returns GDN_ERR_REFUSED after undoing the
 * plan: the pool, reqs and *txn are left as they were ([NATIVE] Results:
 * recovery after abort), so the zero-copy form below keeps writing its
 * checkpoints into the area the locations do not point into.
 * ckpt_tag holds num_layers x B tags (B = decode requests of the plan).
 * kernel_ms (host, 3 floats, or NULL): device time of the verify launches of
 * all layers, of the accept and of the commit with its check, from events
 * on `stream`.
 * Decode requests only: a request list holding a prefill returns
 * GDN_ERR_ARG before anything is planned.  A plan that selects no request,
 * or a call that fails after planning, is undone with gdn_pool_abort (its
 * fresh slots return to the pool) and GDN_ERR_ARG or that call's status is
 * returned.  Blocks the host until the transaction is done (it waits for
 * `stream`, so it cannot be captured into a CUDA graph).
 * Device-detected errors accumulate in *io->dev_status as usual.
 * The two host buffers must be page-locked; when they are mapped into the
 * device address space (so with unified addressing) a one-block kernel moves
 * the tables in and the results out, so neither waits behind a large copy
 * the caller has queued on a copy engine; otherwise cudaMemcpyAsync does.
 */
typedef struct gdn_decode_io {
    int32_t *tables;                  /* device [3][n_reqs+1] */
    const gdn_layer_rows *rows;       /* host array [num_layers] */
    float *pool;
    int64_t slot_stride, layer_stride;
    int32_t num_slots;
    float *ckpt;
    int64_t ckpt_layer_stride;
    uint64_t *ckpt_tag;
    gdn_bf16 *o;
    int64_t o_layer_stride;
    const gdn_bf16 *logits;
    int64_t vocab, logit_row_stride;
    const int32_t *tokens;            /* packed draft ids (device) */
    int32_t *argmax, *accept_len, *bonus, *out_tokens;
    mtp_stats *stats;
    void *workspace;
    size_t workspace_bytes;
    uint32_t *dev_status;
    int32_t *host_tables;             /* page-locked host [3][n_reqs+1] */
    int32_t *host_out;                /* page-locked host [2*n_reqs + row_capacity] */
} gdn_decode_io;

int gdn_decode_transaction(const gdn_dims *dims, int32_t num_layers, int32_t row_capacity,
                           gdn_req *reqs, int32_t n_reqs, const gdn_plan_limits *lim,
                           gdn_pool *pool, gdn_plan *plan, uint32_t *txn,
                           const gdn_decode_io *io, float *kernel_ms, void *stream);

/*
 * gdn_decode_transaction_at -- gdn_decode_transaction over a state arena
 * (the zero-copy commit above): gdn_verify_at_layers reads every start state
 * at arena->arena + loc[l*n_reqs + r] and writes the checkpoints at
 * arena->arena + area_off[(txn + 1) & 1]; gdn_commit_at rewrites loc.
 * io->pool, slot_stride, layer_stride, num_slots and ckpt are not used.
 * Every request must be a decode request selected by the plan (the location
 * table holds one entry per request and layer); otherwise the plan is
 * undone and GDN_ERR_ARG returned.
 */
typedef struct gdn_arena_io {
    float *arena;                     /* device */
    int64_t elems_total;              /* fp32 elements of the arena */
    int64_t *loc;                     /* device [num_layers][n_reqs] element offsets */
    int64_t area_off[2];              /* element offsets of the two checkpoint areas */
} gdn_arena_io;

int gdn_decode_transaction_at(const gdn_dims *dims, int32_t num_layers, int32_t row_capacity,
                              gdn_req *reqs, int32_t n_reqs, const gdn_plan_limits *lim,
                              gdn_pool *pool, gdn_plan *plan, uint32_t *txn,
                              const gdn_decode_io *io, const gdn_arena_io *arena,
                              float *kernel_ms, void *stream);

const char *gdn_status_string(int status);

/* Failure-detection self-test of the chunked prefill: gdn_chunked_prefill
 * (chunk 64) with every wait bounded by limit_ns (1 .. 1e9) of device time,
 * and with the tensor copy of each sequence's last chunk of K and Q
 * withheld, so that the wait for it runs out: every sequence sets
 * GDN_DEV_TIMEOUT and publishes nothing.  d_k = d_v = 128 only (the smaller
 * sizes run no copy-engine wait).  (Test-only; it computes nothing a caller
 * would use.) */
int gdn_selftest_prefill_timeout(const gdn_dims *dims, int32_t nseq, int32_t row_capacity,
                                 const int32_t *cu_seqlens,
                                 const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                                 const float *g, const float *beta,
                                 float *pool_layer, int64_t slot_stride, int32_t num_slots,
                                 const int32_t *src_slot, const int32_t *dst_slot, gdn_bf16 *o,
                                 void *workspace, size_t workspace_bytes,
                                 uint32_t *dev_status, uint64_t limit_ns, void *stream);

/* Failure-detection self-test: a kernel waits on an mbarrier that is never
 * completed, gives up after limit_ns (1 .. 1e9) of device time and sets
 * GDN_DEV_TIMEOUT in *dev_status -- the same bounded wait every kernel here
 * uses for its asynchronous copies and tensor-core operations. */
int gdn_selftest_wait_timeout(uint32_t *dev_status, uint64_t limit_ns, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* GDNSPEC_H */
