// Host-side transaction planner and reference-counted slot pool.
//
// "Run chained MTP drafting in the batch Engine": Summary (per-request draft
// lengths; drafts deferred for a selected transaction that mixes prefill and
// speculative rows, MTP resumed on decode-only transactions), Correctness fix
// (the deferral is applied after paged selection; decode requests still
// advance one token and prefills continue), H200 RC4 evidence (mixed K,
// max-length clamping, cache reuse).  "Native three-step MTP", Results:
// shared-prefix protection, duplicate-slot release, recovery after abort.
//
// Everything here is synchronous host code over caller-owned host arrays.
#include <stdint.h>
#include <string.h>

#include <vector>

#include "gdnspec.h"

namespace {

bool slot_held(const gdn_pool *p, int32_t s) { return s >= 0 && s < p->num_slots && p->refcount[s] > 0; }

void fifo_push_tail(gdn_pool *p, int32_t s) {
    p->free_fifo[(p->free_head + p->free_count) % p->num_slots] = s;
    p->free_count++;
}

void fifo_push_head(gdn_pool *p, int32_t s) {
    p->free_head = (p->free_head + p->num_slots - 1) % p->num_slots;
    p->free_fifo[p->free_head] = s;
    p->free_count++;
}

// Undo fresh-slot reservations in reverse order: the free list regains its
// exact previous order and the counts return to zero.
void unreserve(gdn_pool *p, const std::vector<int32_t> &reserved) {
    for (size_t i = reserved.size(); i-- > 0;) {
        p->refcount[reserved[i]] = 0;
        fifo_push_head(p, reserved[i]);
    }
}

}  // namespace

extern "C" int gdn_pool_init(gdn_pool *pool, int32_t num_slots, int32_t *refcount, int32_t *free_fifo,
                             const int32_t *free_order) {
    if (!pool || !refcount || !free_fifo) return GDN_ERR_NULL;
    if (num_slots <= 0) return GDN_ERR_ARG;
    std::vector<char> seen(size_t(num_slots), 0);
    if (free_order) {
        for (int32_t i = 0; i < num_slots; ++i) {
            const int32_t s = free_order[i];
            if (s < 0 || s >= num_slots || seen[size_t(s)]) return GDN_ERR_ARG;
            seen[size_t(s)] = 1;
        }
    }
    pool->num_slots = num_slots;
    pool->refcount = refcount;
    pool->free_fifo = free_fifo;
    pool->free_head = 0;
    pool->free_count = num_slots;
    for (int32_t i = 0; i < num_slots; ++i) {
        refcount[i] = 0;
        free_fifo[i] = free_order ? free_order[i] : i;
    }
    return GDN_OK;
}

extern "C" int gdn_pool_alloc(gdn_pool *pool, int32_t *slot) {
    if (!pool || !slot) return GDN_ERR_NULL;
    if (pool->free_count == 0) return GDN_ERR_NO_SLOT;
    const int32_t s = pool->free_fifo[pool->free_head];
    pool->free_head = (pool->free_head + 1) % pool->num_slots;
    pool->free_count--;
    pool->refcount[s] = 1;
    *slot = s;
    return GDN_OK;
}

extern "C" int gdn_pool_share(gdn_pool *pool, int32_t slot) {
    if (!pool) return GDN_ERR_NULL;
    if (!slot_held(pool, slot)) return GDN_ERR_ARG;
    pool->refcount[slot]++;
    return GDN_OK;
}

extern "C" int gdn_pool_release(gdn_pool *pool, int32_t slot) {
    if (!pool) return GDN_ERR_NULL;
    if (!slot_held(pool, slot)) return GDN_ERR_ARG;  // includes a second release of a freed slot
    if (--pool->refcount[slot] == 0) fifo_push_tail(pool, slot);
    return GDN_OK;
}

extern "C" int plan_transaction(const gdn_req *reqs, int32_t n, const gdn_plan_limits *lim, gdn_pool *pool,
                                gdn_plan *out) {
    if (!lim || !pool || !out || (n > 0 && !reqs)) return GDN_ERR_NULL;
    if (n < 0 || lim->max_rows < 0 || lim->max_reqs < 0 || lim->k_max < 0 || lim->k_max > GDN_K_MAX)
        return GDN_ERR_ARG;
    if (n > 0 && (!out->k || !out->rows || !out->src || !out->dst || !out->dec_req || !out->dec_cu ||
                  !out->dec_src || !out->dec_dst || !out->pre_req || !out->pre_cu || !out->pre_src ||
                  !out->pre_dst))
        return GDN_ERR_NULL;
    out->n_selected = 0;
    out->plan = GDN_PLAN_RECURRENT;
    out->deferred = 0;
    out->n_decode = out->decode_rows = out->n_prefill = out->prefill_rows = 0;
    for (int32_t i = 0; i < n; ++i) {
        out->k[i] = -1;
        out->rows[i] = 0;
        out->src[i] = -1;
        out->dst[i] = -1;
    }
    if (out->dec_cu) out->dec_cu[0] = 0;
    if (out->pre_cu) out->pre_cu[0] = 0;

    // 1. paged selection, in request order
    int64_t budget = lim->max_rows;
    int32_t nsel = 0;
    for (int32_t i = 0; i < n; ++i) {
        if (nsel >= lim->max_reqs || budget < 1) break;
        const gdn_req &r = reqs[i];
        if (r.slot != -1 && !slot_held(pool, r.slot)) return GDN_ERR_ARG;
        if (r.kind == GDN_REQ_DECODE) {
            if (r.cur_len >= r.max_len || r.k_draft < 0 || r.slot < 0) return GDN_ERR_ARG;
            int64_t K = r.k_draft;
            if (K > lim->k_max) K = lim->k_max;
            if (K > int64_t(r.max_len) - r.cur_len - 1) K = int64_t(r.max_len) - r.cur_len - 1;
            if (K > budget - 1) K = budget - 1;
            if (K < 0) K = 0;
            out->k[i] = int32_t(K);
            out->rows[i] = int32_t(K + 1);
        } else if (r.kind == GDN_REQ_PREFILL) {
            if (r.n_tokens <= 0 || r.cur_len >= r.max_len) return GDN_ERR_ARG;
            int64_t rows = r.n_tokens;
            if (rows > int64_t(r.max_len) - r.cur_len) rows = int64_t(r.max_len) - r.cur_len;
            if (rows > budget) rows = budget;
            out->k[i] = 0;
            out->rows[i] = int32_t(rows);
        } else {
            return GDN_ERR_ARG;
        }
        budget -= out->rows[i];
        ++nsel;
    }
    out->n_selected = nsel;

    // 2. defer drafts when prefill and draft rows share the transaction
    bool has_prefill = false, has_draft = false;
    for (int32_t i = 0; i < nsel; ++i) {
        if (reqs[i].kind == GDN_REQ_PREFILL) has_prefill = true;
        if (reqs[i].kind == GDN_REQ_DECODE && out->k[i] > 0) has_draft = true;
    }
    if (has_prefill && has_draft) {
        for (int32_t i = 0; i < nsel; ++i)
            if (reqs[i].kind == GDN_REQ_DECODE) {
                out->deferred += out->k[i];
                out->k[i] = 0;
                out->rows[i] = 1;
            }
    }
    // 3. plan kind
    out->plan = has_prefill ? GDN_PLAN_CHUNKED : GDN_PLAN_RECURRENT;

    // 4. slots: in place for a slot held once, fresh (copy-on-write) otherwise
    std::vector<int32_t> reserved;
    for (int32_t i = 0; i < nsel; ++i) {
        const int32_t s = reqs[i].slot;
        out->src[i] = s;
        if (s >= 0 && pool->refcount[s] == 1) {
            out->dst[i] = s;
        } else {
            int32_t fresh = -1;
            if (gdn_pool_alloc(pool, &fresh) != GDN_OK) {
                unreserve(pool, reserved);
                return GDN_ERR_NO_SLOT;
            }
            reserved.push_back(fresh);
            out->dst[i] = fresh;
        }
    }
    {
        std::vector<char> used(size_t(pool->num_slots), 0);
        for (int32_t i = 0; i < nsel; ++i) {
            const int32_t d = out->dst[i];
            if (used[size_t(d)]) {
                unreserve(pool, reserved);
                return GDN_ERR_DUP_SLOT;
            }
            used[size_t(d)] = 1;
        }
    }
    // group tables in request order
    for (int32_t i = 0; i < nsel; ++i) {
        if (reqs[i].kind == GDN_REQ_DECODE) {
            const int32_t j = out->n_decode++;
            out->dec_req[j] = i;
            out->dec_src[j] = out->src[i];
            out->dec_dst[j] = out->dst[i];
            out->dec_cu[j + 1] = out->dec_cu[j] + out->rows[i];
            out->decode_rows += out->rows[i];
        } else {
            const int32_t j = out->n_prefill++;
            out->pre_req[j] = i;
            out->pre_src[j] = out->src[i];
            out->pre_dst[j] = out->dst[i];
            out->pre_cu[j + 1] = out->pre_cu[j] + out->rows[i];
            out->prefill_rows += out->rows[i];
        }
    }
    return GDN_OK;
}

extern "C" int gdn_pool_apply(gdn_pool *pool, const gdn_plan *plan, int32_t n) {
    if (!pool || !plan) return GDN_ERR_NULL;
    for (int32_t i = 0; i < n; ++i)
        if (plan->k[i] >= 0 && plan->src[i] >= 0 && plan->dst[i] != plan->src[i]) {
            const int st = gdn_pool_release(pool, plan->src[i]);
            if (st != GDN_OK) return st;
        }
    return GDN_OK;
}

extern "C" int gdn_pool_abort(gdn_pool *pool, const gdn_plan *plan, int32_t n) {
    if (!pool || !plan) return GDN_ERR_NULL;
    for (int32_t i = 0; i < n; ++i)
        if (plan->k[i] >= 0 && plan->dst[i] != plan->src[i]) {
            const int st = gdn_pool_release(pool, plan->dst[i]);
            if (st != GDN_OK) return st;
        }
    return GDN_OK;
}

extern "C" const char *gdn_status_string(int status) {
    switch (status) {
        case GDN_OK: return "ok";
        case GDN_ERR_NULL: return "null pointer";
        case GDN_ERR_SHAPE: return "unsupported shape";
        case GDN_ERR_ARG: return "invalid argument";
        case GDN_ERR_DUP_SLOT: return "duplicate destination slot";
        case GDN_ERR_NO_SLOT: return "no free slot";
        case GDN_ERR_CUDA: return "CUDA error";
        case GDN_ERR_WORKSPACE: return "workspace missing or too small";
        case GDN_ERR_REFUSED: return "transaction refused by a device-side check; nothing committed";
        default: return "unknown status";
    }
}
