// extern "C" entry points of libe0moe: argument validation on the host, then
// the launchers in namespace e0.  Nothing here allocates device memory.
#include <cuda_runtime.h>

#include "e0_common.cuh"
#include "e0_internal.h"

namespace {

inline cudaStream_t cs(e0_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool shape_ok(int n) { return n > 0 && n % 64 == 0 && n <= 2048; }

int check_route(const e0_route_params* rp, int E) {
    if (!rp) return E0_ERR_NULL;
    if (E < 1 || E > E0_MAX_E) return E0_ERR_UNSUPPORTED;
    if (rp->K < 1 || rp->K > E0_MAX_K || rp->K > E) return rp->K > E0_MAX_K ? E0_ERR_UNSUPPORTED : E0_ERR_ARG;
    if (rp->mode == E0_ROUTE_SOFTMAX_TOPK) return E0_OK;
    if (rp->mode != E0_ROUTE_SIGMOID_GROUP) return E0_ERR_ARG;
    const int n = rp->n_groups, G = rp->topk_groups;
    if (n < 1 || G < 1 || G > n || E % n != 0) return E0_ERR_ARG;
    if (n > 32) return E0_ERR_UNSUPPORTED;
    if (rp->K > G * (E / n)) return E0_ERR_ARG;
    return E0_OK;
}

int check_pool(const e0_slot_pool* p) {
    if (!p) return E0_ERR_NULL;
    if (!p->data || !p->slot_table) return E0_ERR_NULL;
    if (!shape_ok(p->H) || !shape_ok(p->I)) return E0_ERR_UNSUPPORTED;
    if (p->E < 1 || p->E > E0_MAX_E || p->n_slots < 1) return E0_ERR_ARG;
    return E0_OK;
}

int check_shared(const e0_shared_expert* sh) {
    if (!sh) return E0_OK;
    if (!sh->data) return E0_ERR_NULL;
    const bool any = sh->A_gate || sh->B_gate || sh->A_up || sh->B_up || sh->A_down || sh->B_down;
    const bool all = sh->A_gate && sh->B_gate && sh->A_up && sh->B_up && sh->A_down && sh->B_down;
    if (any && !all) return E0_ERR_NULL;
    if (all && (sh->rank < 1 || sh->rank > E0_MAX_LORA_RANK)) return E0_ERR_UNSUPPORTED;
    return E0_OK;
}

int check_head(const e0_prerouter* h) {
    if (!h) return E0_OK;
    if (!h->fc1 || !h->fc2 || !h->lres) return E0_ERR_NULL;
    if (!shape_ok(h->H) || !shape_ok(h->hidden)) return E0_ERR_UNSUPPORTED;
    if (h->E < 1 || h->E > E0_MAX_E) return E0_ERR_UNSUPPORTED;
    if (((size_t)(h->H + 2 * h->E) * 2) % 16 != 0) return E0_ERR_UNSUPPORTED;
    return E0_OK;
}

}  // namespace

extern "C" {

size_t e0_slot_bytes(int H, int I) {
    if (!shape_ok(H) || !shape_ok(I)) return 0;
    return e0::slot_bytes(H, I);
}

size_t e0_workspace_size(int op, int T, int H, int I, int E, int K) {
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || K <= 0) return 0;
    switch (op) {
        case 0: return e0::block_ws_bytes(T, H, I, E, K, E0_MAX_LORA_RANK, 0);
        case 1: return e0::head_ws_bytes(T, H, I, E, K);
        case 2: return e0::prefill_ws_bytes(T, H, I, E, K);
        default: return 0;
    }
}

int e0_pack_experts(const e0_expert_q* src, int n, const e0_slot_pool* dst, const int32_t* dst_slots,
                    const int32_t* expert_ids, e0_stream_t stream) {
    if (n == 0) return E0_OK;
    if (!src || !dst || !dst_slots) return E0_ERR_NULL;
    if (n < 0) return E0_ERR_ARG;
    if (!dst->data) return E0_ERR_NULL;
    if (!shape_ok(dst->H) || !shape_ok(dst->I)) return E0_ERR_UNSUPPORTED;
    if (expert_ids && (!dst->slot_table)) return E0_ERR_NULL;
    for (int i = 0; i < n; ++i) {
        const e0_expert_q& e = src[i];
        if (!e.gate.codes || !e.gate.scale || !e.gate.bias || !e.up.codes || !e.up.scale || !e.up.bias ||
            !e.down.codes || !e.down.scale || !e.down.bias)
            return E0_ERR_NULL;
        if (dst_slots[i] < 0 || dst_slots[i] >= dst->n_slots) return E0_ERR_ARG;
        if (expert_ids && (expert_ids[i] < 0 || expert_ids[i] >= dst->E)) return E0_ERR_ARG;
        // 16-byte chunks are copied: code rows must be 16-byte aligned
        if (((uintptr_t)e.gate.codes | (uintptr_t)e.up.codes | (uintptr_t)e.down.codes) & 15) return E0_ERR_ARG;
    }
    return e0::pack_experts(src, n, dst, dst_slots, expert_ids, cs(stream));
}

int e0_slot_update(const e0_slot_pool* pool, const int32_t* d_inds_next, int n_next, const int32_t* d_inds_cur,
                   int n_cur, const uint8_t* bank, uint32_t* d_status, e0_stream_t stream) {
    int rc = check_pool(pool);
    if (rc) return rc;
    if (!pool->occupant) return E0_ERR_NULL;
    if (n_next < 0 || n_cur < 0) return E0_ERR_ARG;
    if (n_next > E0_MAX_T_DECODE * E0_MAX_K || n_cur > E0_MAX_T_DECODE * E0_MAX_K) return E0_ERR_UNSUPPORTED;
    if (n_next == 0) return E0_OK;
    if (!d_inds_next || !bank) return E0_ERR_NULL;
    if (n_cur > 0 && !d_inds_cur) return E0_ERR_NULL;
    if (((uintptr_t)bank | (uintptr_t)pool->data) & 15) return E0_ERR_ARG;
    return e0::slot_update(pool, d_inds_next, n_next, n_cur ? d_inds_cur : nullptr, n_cur, bank, d_status,
                           cs(stream));
}

int e0_route_softmax_topk(const float* logits, int T, int E, int K, int32_t* inds, float* w, uint32_t* d_status,
                          e0_stream_t stream) {
    if (T < 0) return E0_ERR_ARG;
    e0_route_params rp = {E0_ROUTE_SOFTMAX_TOPK, K, 1, 1, 1.f, nullptr};
    int rc = check_route(&rp, E);
    if (rc) return rc;
    if (T == 0) return E0_OK;
    if (!logits || !inds || !w) return E0_ERR_NULL;
    return e0::route(logits, T, E, &rp, inds, w, d_status, cs(stream));
}

int e0_route_sigmoid_group(const float* logits, int T, int E, int n_groups, int topk_groups, int K, float s,
                           int32_t* inds, float* w, uint32_t* d_status, e0_stream_t stream) {
    if (T < 0) return E0_ERR_ARG;
    e0_route_params rp = {E0_ROUTE_SIGMOID_GROUP, K, n_groups, topk_groups, s, nullptr};
    int rc = check_route(&rp, E);
    if (rc) return rc;
    if (T == 0) return E0_OK;
    if (!logits || !inds || !w) return E0_ERR_NULL;
    return e0::route(logits, T, E, &rp, inds, w, d_status, cs(stream));
}

int e0_rmsnorm(const float* r, int T, int H, float eps, float* h, e0_stream_t stream) {
    if (T < 0 || H <= 0 || !(eps >= 0.f)) return E0_ERR_ARG;
    if (T == 0) return E0_OK;
    if (!r || !h) return E0_ERR_NULL;
    return e0::rmsnorm(r, T, H, eps, h, cs(stream));
}

int e0_moe_block_forward(const float* x, int T, const e0_slot_pool* pool, const uint16_t* W_router,
                         const e0_route_params* rp, const int32_t* inds_in, const float* w_in,
                         const e0_shared_expert* shared, float* y, int32_t* inds_out, float* w_out, void* ws,
                         size_t ws_bytes, uint32_t* d_status, e0_stream_t stream) {
    int rc = check_pool(pool);
    if (rc) return rc;
    if ((rc = check_route(rp, pool->E))) return rc;
    if ((rc = check_shared(shared))) return rc;
    if (T < 0) return E0_ERR_ARG;
    if (T > E0_MAX_T_DECODE) return E0_ERR_UNSUPPORTED;
    if (T == 0) return E0_OK;
    if (!x || !y || !ws) return E0_ERR_NULL;
    if ((inds_in == nullptr) != (w_in == nullptr)) return E0_ERR_NULL;
    if (!inds_in && !W_router) return E0_ERR_NULL;
    if (ws_bytes < e0_workspace_size(0, T, pool->H, pool->I, pool->E, rp->K)) return E0_ERR_ARG;
    if (((uintptr_t)ws & 255) || ((uintptr_t)x & 15) || ((uintptr_t)pool->data & 15)) return E0_ERR_ARG;
    return e0::moe_block_forward(x, T, pool, W_router, rp, inds_in, w_in, shared, y, inds_out, w_out, ws, d_status,
                                 cs(stream));
}

int e0_prerouter_forward(const float* h, int T, const int32_t* inds_cur, const int32_t* inds_prev,
                         const e0_prerouter* head, const e0_route_params* rp, float* logits_out, int32_t* inds_next,
                         float* w_next, void* ws, size_t ws_bytes, uint32_t* d_status, e0_stream_t stream) {
    if (!head) return E0_ERR_NULL;
    int rc = check_head(head);
    if (rc) return rc;
    if ((rc = check_route(rp, head->E))) return rc;
    if (T < 0) return E0_ERR_ARG;
    if (T > E0_MAX_T_DECODE) return E0_ERR_UNSUPPORTED;
    if (T == 0) return E0_OK;
    if (!h || !inds_cur || !inds_next || !w_next || !ws) return E0_ERR_NULL;
    if (ws_bytes < e0_workspace_size(1, T, head->H, head->hidden, head->E, rp->K)) return E0_ERR_ARG;
    if (((uintptr_t)ws & 255) || ((uintptr_t)h & 15)) return E0_ERR_ARG;
    return e0::prerouter_forward(h, T, inds_cur, inds_prev, head, rp, logits_out, inds_next, w_next, ws, d_status,
                                 cs(stream));
}

size_t e0_stack_workspace_size(int L, int H, int I, int E, int K, int head_hidden) {
    if (L < 1 || !shape_ok(H) || !shape_ok(I) || E < 1 || E > E0_MAX_E || K < 1 || K > E0_MAX_K) return 0;
    if (head_hidden < 0 || head_hidden > 2048) return 0;
    return e0::stack_ws_bytes(L, H, I, E, K, head_hidden);
}

int e0_stack_prepare(const e0_stack_layer* layers, int L, int H, int I, int E, const e0_route_params* rp, void* ws,
                     size_t ws_bytes, e0_stream_t stream) {
    if (!layers || !ws) return E0_ERR_NULL;
    if (L < 1) return E0_ERR_ARG;
    int rc = check_route(rp, E);
    if (rc) return rc;
    if (!shape_ok(H) || !shape_ok(I)) return E0_ERR_UNSUPPORTED;
    int hidden = 0;
    for (int l = 0; l < L; ++l) {
        const e0_stack_layer& s = layers[l];
        if ((rc = check_pool(&s.pool))) return rc;
        if (s.pool.H != H || s.pool.I != I || s.pool.E != E) return E0_ERR_ARG;
        if (!s.W_router) return E0_ERR_NULL;
        if ((rc = check_shared(s.shared))) return rc;
        if ((rc = check_head(s.head))) return rc;
        if (s.head && (s.head->H != H || s.head->E != E)) return E0_ERR_ARG;
        if (s.head && s.head->hidden > hidden) hidden = s.head->hidden;
        if (s.consumer && (l == 0 || !layers[l - 1].head)) return E0_ERR_ARG;
    }
    if (ws_bytes < e0_stack_workspace_size(L, H, I, E, rp->K, hidden)) return E0_ERR_ARG;
    if ((uintptr_t)ws & 255) return E0_ERR_ARG;
    return e0::stack_prepare(layers, L, H, I, E, rp, ws, cs(stream));
}

int e0_stack_step(const float* x, float* r_out, void* ws, const e0_stack_trace* trace, int impl, uint32_t* d_status,
                  e0_stream_t stream) {
    if (!x || !r_out || !ws) return E0_ERR_NULL;
    if (impl < 0 || impl > 3) return E0_ERR_ARG;
    if (!e0::stack_known(ws)) return E0_ERR_ARG;
    return e0::stack_step(x, r_out, ws, trace, impl, d_status, cs(stream));
}

int e0_prefill_sort(const int32_t* inds, int T, int K, int E, int32_t* counts, int32_t* offsets, int32_t* perm,
                    void* ws, size_t ws_bytes, e0_stream_t stream) {
    if (T < 0 || K < 1 || K > E0_MAX_K || E < 1 || E > E0_MAX_E) return E0_ERR_ARG;
    if (!counts || !offsets) return E0_ERR_NULL;
    if (T > 0 && (!inds || !perm || !ws)) return E0_ERR_NULL;
    if (ws_bytes < e0_workspace_size(2, T, 64, 64, E, K)) return E0_ERR_ARG;
    return e0::prefill_sort(inds, T, K, E, counts, offsets, perm, ws, cs(stream));
}

int e0_moe_prefill_forward(const uint16_t* X, int T, const e0_slot_pool* bank, const uint16_t* W_router,
                           const e0_route_params* rp, float* Y, int32_t* inds_out, float* w_out, void* ws,
                           size_t ws_bytes, uint32_t* d_status, e0_stream_t stream) {
    int rc = check_pool(bank);
    if (rc) return rc;
    if ((rc = check_route(rp, bank->E))) return rc;
    if (T < 0) return E0_ERR_ARG;
    if (T == 0) return E0_OK;
    if (!X || !W_router || !Y || !ws) return E0_ERR_NULL;
    if (ws_bytes < e0_workspace_size(2, T, bank->H, bank->I, bank->E, rp->K)) return E0_ERR_ARG;
    if (((uintptr_t)ws & 255) || ((uintptr_t)X & 15) || ((uintptr_t)W_router & 15)) return E0_ERR_ARG;
    return e0::moe_prefill_forward(X, T, bank, W_router, rp, Y, inds_out, w_out, ws, d_status, cs(stream));
}

int e0_stack_step_range(const float* x, float* r_out, void* ws, int layer_begin, int layer_end,
                        const e0_stack_trace* trace, uint32_t* d_status, e0_stream_t stream) {
    if (!ws) return E0_ERR_NULL;
    if (!e0::stack_known(ws)) return E0_ERR_ARG;
    if (layer_begin == 0 && !x) return E0_ERR_NULL;
    return e0::stack_step_range(x, r_out, ws, layer_begin, layer_end, trace, d_status, cs(stream));
}

int e0_stack_update_layers(void* ws, const e0_stack_layer* layers, int L, e0_stream_t stream) {
    if (!ws || !layers) return E0_ERR_NULL;
    if (!e0::stack_known(ws)) return E0_ERR_ARG;
    for (int l = 0; l < L; ++l) {
        const int rc = check_pool(&layers[l].pool);
        if (rc != E0_OK) return rc;
    }
    return e0::stack_update_layers(ws, layers, L, cs(stream));
}

int e0_stack_prefetch_experts(void* ws, int layer, int t_next, const e0_slot_pool* pool, const uint8_t* bank,
                              uint32_t* d_status, e0_stream_t stream) {
    if (!ws || !pool || !bank) return E0_ERR_NULL;
    if (!e0::stack_known(ws)) return E0_ERR_ARG;
    const int rc = check_pool(pool);
    if (rc != E0_OK) return rc;
    return e0::stack_prefetch_experts(ws, layer, t_next, pool, bank, d_status, cs(stream));
}

int e0_stack_prefetch_experts_batch(void* ws, const int32_t* layers, int n, int t_next, const e0_slot_pool* pools,
                                    const uint8_t* const* banks, uint32_t* d_status, e0_stream_t stream) {
    if (!ws || (n > 0 && (!layers || !pools || !banks))) return E0_ERR_NULL;
    if (!e0::stack_known(ws)) return E0_ERR_ARG;
    for (int i = 0; i < n; ++i) {
        if (!banks[i]) return E0_ERR_NULL;
        const int rc = check_pool(&pools[i]);
        if (rc != E0_OK) return rc;
        // the layers' pools must be disjoint: their copies run at the same time
        for (int j = 0; j < i; ++j)
            if (pools[j].data == pools[i].data || pools[j].slot_table == pools[i].slot_table) return E0_ERR_ARG;
    }
    return e0::stack_prefetch_experts_batch(ws, layers, n, t_next, pools, banks, d_status, cs(stream));
}

int e0_stack_prefetch_experts_cached_batch(void* ws, const int32_t* layers, int n, int t_next,
                                           const e0_slot_pool* pools, const uint8_t* const* banks,
                                           const e0_expert_cache* cache, uint32_t* d_status, e0_stream_t stream) {
    if (!ws || !cache || (n > 0 && (!layers || !pools || !banks))) return E0_ERR_NULL;
    if (!e0::stack_known(ws)) return E0_ERR_ARG;
    if (cache->capacity < 0 || cache->n_keys < 1) return E0_ERR_ARG;
    if (!cache->key || !cache->stamp || !cache->map || !cache->counters || (cache->capacity > 0 && !cache->data))
        return E0_ERR_NULL;
    for (int i = 0; i < n; ++i) {
        if (!banks[i]) return E0_ERR_NULL;
        const int rc = check_pool(&pools[i]);
        if (rc != E0_OK) return rc;
        for (int j = 0; j < i; ++j)
            if (pools[j].data == pools[i].data || pools[j].slot_table == pools[i].slot_table) return E0_ERR_ARG;
    }
    return e0::stack_prefetch_experts_cached_batch(ws, layers, n, t_next, pools, banks, cache, d_status, cs(stream));
}

int e0_stack_prefetch_experts_cached(void* ws, int layer, int t_next, const e0_slot_pool* pool, const uint8_t* bank,
                                     const e0_expert_cache* cache, uint32_t* d_status, e0_stream_t stream) {
    if (!ws || !pool || !bank || !cache) return E0_ERR_NULL;
    if (!e0::stack_known(ws)) return E0_ERR_ARG;
    const int rc = check_pool(pool);
    if (rc != E0_OK) return rc;
    if (cache->capacity < 0 || cache->n_keys < 1) return E0_ERR_ARG;
    if (!cache->key || !cache->stamp || !cache->map || !cache->counters || !cache->scratch ||
        (cache->capacity > 0 && !cache->data))
        return E0_ERR_NULL;
    return e0::stack_prefetch_experts_cached(ws, layer, t_next, pool, bank, cache, d_status, cs(stream));
}

int e0_selftest_bounded_wait(const uint32_t* flag, uint32_t limit_us, uint32_t* d_status, e0_stream_t stream) {
    if (!flag || !d_status) return E0_ERR_NULL;
    if (limit_us == 0 || limit_us > E0_SELFTEST_MAX_WAIT_US) return E0_ERR_ARG;
    return e0::selftest_bounded_wait(flag, limit_us, d_status, cs(stream));
}

int e0_read_status(const uint32_t* d_status, uint32_t* h_out, e0_stream_t stream) {
    if (!d_status || !h_out) return E0_ERR_NULL;
    if (cudaMemcpyAsync(h_out, d_status, sizeof(uint32_t), cudaMemcpyDeviceToHost, cs(stream)) != cudaSuccess)
        return E0_ERR_CUDA;
    return cudaStreamSynchronize(cs(stream)) == cudaSuccess ? E0_OK : E0_ERR_CUDA;
}

const char* e0_status_string(int code) {
    switch (code) {
        case E0_OK: return "ok";
        case E0_ERR_ARG: return "invalid argument (shape, size or option)";
        case E0_ERR_NULL: return "a required pointer is NULL";
        case E0_ERR_UNSUPPORTED: return "valid but unsupported by these kernels";
        case E0_ERR_CUDA: return "CUDA launch or copy error";
        default: return "unknown status code";
    }
}

}  // extern "C"

namespace e0 {
size_t slot_bytes(int H, int I) { return SlotLayout{H, I}.bytes(); }
}  // namespace e0
