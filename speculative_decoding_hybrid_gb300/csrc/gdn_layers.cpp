// Multi-layer issue of the per-layer verify calls: one host call walks the
// layers in order and makes the same gdn_verify / gdn_verify_replay calls a
// caller would make layer by layer (same kernels, same arguments, same
// stream), so a step that holds every layer's inputs pays one host call
// instead of one per layer.
#include "gdnspec.h"

#include <cstdint>

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
        const int st = gdn_verify(dims, B, row_capacity, cu_rows, x.q, x.k, x.v, x.g, x.beta,
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
        const int st = gdn_verify_replay(dims, B, row_capacity, cu_rows, x.q, x.k, x.v, x.g, x.beta, prev_capacity,
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
        const int st = gdn_verify_at(dims, B, row_capacity, cu_rows, x.q, x.k, x.v, x.g, x.beta, state_base,
                                     state_elems_total, src_off + int64_t(l) * B,
                                     ckpt + int64_t(l) * ckpt_layer_stride, ckpt_tag + int64_t(l) * B, txn,
                                     o + int64_t(l) * o_layer_stride, dev_status, stream);
        if (st != GDN_OK) return st;
    }
    return GDN_OK;
}
