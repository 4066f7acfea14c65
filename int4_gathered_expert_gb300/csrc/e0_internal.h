// Host-side entry points shared between the translation units of libe0moe.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/e0moe.h"

namespace e0 {

int num_sms();
int selftest_bounded_wait(const uint32_t* flag, uint32_t limit_us, uint32_t* st, cudaStream_t s);
size_t slot_bytes(int H, int I);

int pack_experts(const e0_expert_q* src, int n, const e0_slot_pool* dst, const int32_t* dst_slots,
                 const int32_t* expert_ids, cudaStream_t s);
int slot_update(const e0_slot_pool* p, const int32_t* next, int n_next, const int32_t* cur, int n_cur,
                const uint8_t* bank, uint32_t* st, cudaStream_t s, int grid = 0);
int stack_step_range(const float* x, float* r_out, void* ws, int lb, int le, const e0_stack_trace* trace, uint32_t* st,
                     cudaStream_t s);
int stack_update_layers(void* ws, const e0_stack_layer* layers, int L, cudaStream_t s);
int stack_prefetch_experts(void* ws, int layer, int t_next, const e0_slot_pool* pool, const uint8_t* bank, uint32_t* st,
                           cudaStream_t s);
int stack_prefetch_experts_batch(void* ws, const int32_t* layers, int n, int t_next, const e0_slot_pool* pools,
                                 const uint8_t* const* banks, uint32_t* st, cudaStream_t s);
int stack_prefetch_experts_cached_batch(void* ws, const int32_t* layers, int n, int t_next, const e0_slot_pool* pools,
                                        const uint8_t* const* banks, const e0_expert_cache* c, uint32_t* st,
                                        cudaStream_t s);
int stack_prefetch_experts_cached(void* ws, int layer, int t_next, const e0_slot_pool* pool, const uint8_t* bank,
                                  const e0_expert_cache* cache, uint32_t* st, cudaStream_t s);
int route(const float* logits, int T, int E, const e0_route_params* rp, int32_t* inds, float* w, uint32_t* st,
          cudaStream_t s);
int rmsnorm(const float* r, int T, int H, float eps, float* h, cudaStream_t s);

size_t block_ws_bytes(int T, int H, int I, int E, int K, int rank, int hidden);
int moe_block_forward(const float* x, int T, const e0_slot_pool* pool, const uint16_t* W_r,
                      const e0_route_params* rp, const int32_t* inds_in, const float* w_in,
                      const e0_shared_expert* sh, float* y, int32_t* inds_out, float* w_out, void* ws,
                      uint32_t* st, cudaStream_t s);

size_t head_ws_bytes(int T, int H, int hidden, int E, int K);
int prerouter_forward(const float* h, int T, const int32_t* inds_cur, const int32_t* inds_prev,
                      const e0_prerouter* head, const e0_route_params* rp, float* logits_out, int32_t* inds_next,
                      float* w_next, void* ws, uint32_t* st, cudaStream_t s);

size_t stack_ws_bytes(int L, int H, int I, int E, int K, int hidden);
int stack_prepare(const e0_stack_layer* layers, int L, int H, int I, int E, const e0_route_params* rp, void* ws,
                  cudaStream_t s);
bool stack_known(const void* ws);
int stack_step(const float* x, float* r_out, void* ws, const e0_stack_trace* trace, int impl, uint32_t* st,
               cudaStream_t s);

size_t prefill_ws_bytes(int T, int H, int I, int E, int K);
int prefill_sort(const int32_t* inds, int T, int K, int E, int32_t* counts, int32_t* offsets, int32_t* perm,
                 void* ws, cudaStream_t s);
int moe_prefill_forward(const uint16_t* X, int T, const e0_slot_pool* bank, const uint16_t* W_r,
                        const e0_route_params* rp, float* Y, int32_t* inds_out, float* w_out, void* ws,
                        uint32_t* st, cudaStream_t s);

}  // namespace e0
