// Decode path of the int4 gathered-expert MoE block: kernels and the C entry
// points for packing, slot update, routing, RMSNorm, the MoE block, the
// prerouter head and the whole-token decode stack.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <vector>

#include "e0_decode.cuh"
#include "e0_internal.h"

namespace e0 {

constexpr int PHASE_THREADS = 256;
constexpr uint32_t BARRIER_SPIN_LIMIT = 1u << 22;

// ================================================================== packing

__global__ void k_pack_expert(e0_expert_q src, uint8_t* dst, int H, int I, int32_t* table, int32_t* occupant,
                              int eid, int slot) {
    const SlotLayout sl{H, I};
    const int GH = H / GROUP, GI = I / GROUP;
    const size_t n_gu = (size_t)I * H / 16;            // 16-byte chunks of gate/up codes
    const size_t n_dn = (size_t)H * I / 2 / 16;        // down codes
    const size_t n_gsb = (size_t)I * GH * 2;           // gate/up scale-bias pairs
    const size_t n_dsb = (size_t)H * GI;               // down scale-bias pairs
    const size_t total = n_gu + n_dn + n_gsb + n_dsb;
    const size_t row16 = (size_t)H / 16;               // chunks per interleaved gate+up row
    for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q < total; q += (size_t)gridDim.x * blockDim.x) {
        if (q < n_gu) {
            const size_t i = q / row16, c = q % row16;
            const size_t half = row16 / 2;
            const uint8_t* s = c < half ? src.gate.codes + i * (H / 2) + c * 16 : src.up.codes + i * (H / 2) + (c - half) * 16;
            *reinterpret_cast<uint4*>(dst + i * H + c * 16) = interleave16(*reinterpret_cast<const uint4*>(s));
        } else if (q < n_gu + n_dn) {
            // chunk (j, c) = row j, inputs 32c..32c+31, at its row-block offset
            const size_t q2 = q - n_gu, c = q2 / H, j = q2 % H;
            *reinterpret_cast<uint4*>(dst + sl.down_code_off((int)j, (int)c)) =
                interleave16(*reinterpret_cast<const uint4*>(src.down.codes + j * (I / 2) + c * 16));
        } else if (q < n_gu + n_dn + n_gsb) {
            const size_t p = q - n_gu - n_dn;
            const size_t i = p / (2 * GH), which = (p / GH) % 2, g = p % GH;
            const e0_qtensor& qt = which ? src.up : src.gate;
            const uint32_t v = (uint32_t)qt.scale[i * GH + g] | ((uint32_t)qt.bias[i * GH + g] << 16);
            *reinterpret_cast<uint32_t*>(dst + sl.gu_sb() + p * 4) = v;
        } else {
            // word (j, g) = group g of row j, at its row-block offset
            const size_t p = q - n_gu - n_dn - n_gsb, g = p / H, j = p % H;
            const uint32_t v = (uint32_t)src.down.scale[j * GI + g] | ((uint32_t)src.down.bias[j * GI + g] << 16);
            *reinterpret_cast<uint32_t*>(dst + sl.down_sb_off((int)j, (int)g)) = v;
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && table != nullptr && eid >= 0) {
        table[eid] = slot;
        if (occupant) occupant[slot] = eid;
    }
}

// ================================================================== slot update

struct SlotPlan {
    int n;
    int e[E0_MAX_T_DECODE * E0_MAX_K];
    int s[E0_MAX_T_DECODE * E0_MAX_K];
    uint32_t status;
};

// Single thread: the copies that bring every expert of `next` into the pool.
E0_DEV void slot_plan(const int32_t* table, const int32_t* occupant, int n_slots, int E, const int32_t* next,
                      int n_next, const int32_t* cur, int n_cur, SlotPlan* P, uint32_t* prot /*(n_slots+31)/32*/) {
    const int nw = (n_slots + 31) / 32;
    for (int i = 0; i < nw; ++i) prot[i] = 0;
    P->n = 0;
    P->status = 0;
    for (int pass = 0; pass < 2; ++pass) {
        const int32_t* v = pass ? cur : next;
        const int nv = pass ? n_cur : n_next;
        for (int i = 0; v && i < nv; ++i) {
            const int e = v[i];
            if (e < 0 || e >= E) continue;
            const int s = table[e];
            if (s >= 0 && s < n_slots) prot[s >> 5] |= 1u << (s & 31);
        }
    }
    int cursor = 0;
    for (int i = 0; i < n_next; ++i) {
        const int e = next[i];
        if (e < 0 || e >= E) {
            P->status |= E0_ST_BAD_EXPERT;
            continue;
        }
        bool dup = false;
        for (int j = 0; j < i; ++j) dup |= next[j] == e;
        if (dup || table[e] >= 0) continue;
        while (cursor < n_slots && ((prot[cursor >> 5] >> (cursor & 31)) & 1u)) ++cursor;
        if (cursor >= n_slots) {
            P->status |= E0_ST_POOL_FULL;
            continue;
        }
        prot[cursor >> 5] |= 1u << (cursor & 31);
        P->e[P->n] = e;
        P->s[P->n] = cursor;
        P->n++;
    }
    (void)occupant;
}

__global__ void k_slot_copy(const int32_t* table, const int32_t* occupant, uint8_t* pool, int n_slots, int E,
                            const int32_t* next, int n_next, const int32_t* cur, int n_cur, const uint8_t* bank,
                            size_t sbytes) {
    __shared__ SlotPlan P;
    __shared__ uint32_t prot[E0_MAX_E / 32];
    if (threadIdx.x == 0) slot_plan(table, occupant, n_slots, E, next, n_next, cur, n_cur, &P, prot);
    __syncthreads();
    const size_t chunks = sbytes / 16;
    const size_t total = chunks * P.n;
    // four 16-byte loads in flight per thread (the bank may be host memory)
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t q0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q0 < total; q0 += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t q = q0 + u * stride;
            if (q < total)
                v[u] = *reinterpret_cast<const uint4*>(bank + (size_t)P.e[q / chunks] * sbytes + (q % chunks) * 16);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t q = q0 + u * stride;
            if (q < total) *reinterpret_cast<uint4*>(pool + (size_t)P.s[q / chunks] * sbytes + (q % chunks) * 16) = v[u];
        }
    }
}

__global__ void k_slot_commit(int32_t* table, int32_t* occupant, int n_slots, int E, const int32_t* next, int n_next,
                              const int32_t* cur, int n_cur, uint32_t* st) {
    __shared__ SlotPlan P;
    __shared__ uint32_t prot[E0_MAX_E / 32];
    if (threadIdx.x != 0) return;
    slot_plan(table, occupant, n_slots, E, next, n_next, cur, n_cur, &P, prot);
    for (int c = 0; c < P.n; ++c) {
        const int s = P.s[c], e = P.e[c];
        const int old = occupant[s];
        if (old >= 0 && old < E && table[old] == s) table[old] = -1;
        occupant[s] = e;
        table[e] = s;
    }
    if (P.status) set_status(st, P.status);
}

// Several layers' slot updates in two launches: the copy kernel's blocks come
// in groups of `per`, group i updating layer i's pool (each block plans its
// layer's copies itself, as k_slot_copy does); the commit kernel has one block
// per layer.
struct PrefetchLayer {
    int32_t* table;
    int32_t* occupant;
    uint8_t* data;
    const uint8_t* bank;
    const int32_t* next;
    int32_t n_slots, E, layer, pad;
};
constexpr int PREFETCH_MAX_LAYERS = 64;
struct PrefetchBatch {
    PrefetchLayer l[PREFETCH_MAX_LAYERS];
    int32_t n, K, per;
    uint64_t sbytes;
};

__global__ void k_slot_copy_batch(const __grid_constant__ PrefetchBatch B) {
    __shared__ SlotPlan P;
    __shared__ uint32_t prot[E0_MAX_E / 32];
    const int li = blockIdx.x / B.per, b = blockIdx.x % B.per;
    const PrefetchLayer& L = B.l[li];
    if (threadIdx.x == 0) slot_plan(L.table, L.occupant, L.n_slots, L.E, L.next, B.K, nullptr, 0, &P, prot);
    __syncthreads();
    const size_t chunks = B.sbytes / 16;
    const size_t total = chunks * P.n;
    // four 16-byte loads in flight per thread (the bank may be host memory)
    const size_t stride = (size_t)B.per * blockDim.x;
    for (size_t q0 = (size_t)b * blockDim.x + threadIdx.x; q0 < total; q0 += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t q = q0 + u * stride;
            if (q < total)
                v[u] = *reinterpret_cast<const uint4*>(L.bank + (size_t)P.e[q / chunks] * B.sbytes + (q % chunks) * 16);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t q = q0 + u * stride;
            if (q < total) *reinterpret_cast<uint4*>(L.data + (size_t)P.s[q / chunks] * B.sbytes + (q % chunks) * 16) = v[u];
        }
    }
}

__global__ void k_slot_commit_batch(const __grid_constant__ PrefetchBatch B, uint32_t* st) {
    __shared__ SlotPlan P;
    __shared__ uint32_t prot[E0_MAX_E / 32];
    if (threadIdx.x != 0) return;
    const PrefetchLayer& L = B.l[blockIdx.x];
    slot_plan(L.table, L.occupant, L.n_slots, L.E, L.next, B.K, nullptr, 0, &P, prot);
    for (int c = 0; c < P.n; ++c) {
        const int s2 = P.s[c], e = P.e[c];
        const int old = L.occupant[s2];
        if (old >= 0 && old < L.E && L.table[old] == s2) L.table[old] = -1;
        L.occupant[s2] = e;
        L.table[e] = s2;
    }
    if (P.status) set_status(st, P.status);
}

// ================================================================== cross-layer expert cache

// A plan: [0] n copies, then per copy i (4 ints at 4 + 4 i): expert, slot,
// source entry (-1: the bank), cache entry to fill (-1: none).
constexpr int CACHE_PLAN_INTS = 4 + 4 * E0_MAX_K;

// One layer's copies through the cache, planned by one warp (lane 0 keeps the
// bookkeeping).  Entries stamped after `fresh` were used earlier in the same
// launch (as a source or as a fill) and are never evicted: the copies of one
// launch run at the same time, so an entry one of them reads or writes must
// not become another's target.  With every entry taken the expert is copied
// from the bank without being cached.
E0_DEV void cache_plan_layer(const int32_t* table, const int32_t* occupant, int n_slots, int E, const int32_t* next,
                             int n_next, int layer, const e0_expert_cache& c, int32_t* plan, uint32_t& clock,
                             uint32_t fresh, SlotPlan& P, uint32_t* prot, int lane) {
    if (lane == 0) slot_plan(table, occupant, n_slots, E, next, n_next, nullptr, 0, &P, prot);
    __syncwarp();
    int n = 0;
    for (int i = 0; i < P.n; ++i) {
        const int key = layer * E + P.e[i];
        int src = -1, fill = -1;
        const int hit = (key >= 0 && key < c.n_keys) ? c.map[key] : -1;
        if (hit >= 0 && hit < c.capacity) {
            src = hit;
            if (lane == 0) {
                c.stamp[hit] = ++clock;
                c.counters[1] += 1;
            }
        } else {
            if (lane == 0) c.counters[2] += 1;
            if (c.capacity > 0 && key >= 0 && key < c.n_keys) {
                // least recently used entry not used in this launch (an empty
                // one first: stamp 0), the warp scanning a strided share each,
                // ties to the lower entry
                uint32_t best = 0xffffffffu;
                int bi = 0x7fffffff;
                for (int j = lane; j < c.capacity; j += 32) {
                    const uint32_t sj = c.stamp[j];
                    if (sj <= fresh && sj < best) {
                        best = sj;
                        bi = j;
                    }
                }
#pragma unroll
                for (int o = 16; o; o >>= 1) {
                    const uint32_t ob = __shfl_xor_sync(0xffffffffu, best, o);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                    if (ob < best || (ob == best && oi < bi)) {
                        best = ob;
                        bi = oi;
                    }
                }
                if (bi < c.capacity) {
                    fill = bi;
                    if (lane == 0) {
                        const int old = c.key[fill];
                        if (old >= 0 && old < c.n_keys) {
                            c.map[old] = -1;
                            c.counters[3] += 1;
                        }
                        c.key[fill] = key;
                        c.map[key] = fill;
                        c.stamp[fill] = ++clock;
                    }
                }
                __syncwarp();
            }
        }
        if (lane == 0) {
            plan[4 + 4 * n + 0] = P.e[i];
            plan[4 + 4 * n + 1] = P.s[i];
            plan[4 + 4 * n + 2] = src;
            plan[4 + 4 * n + 3] = fill;
        }
        ++n;
        __syncwarp();  // lane 0's bookkeeping is seen by every lane's next scan
    }
    if (lane == 0) plan[0] = n;
}

// One layer's plan into cache->scratch; the copy kernel and the commit
// follow in stream order.
__global__ void k_cache_plan(const int32_t* table, const int32_t* occupant, int n_slots, int E, const int32_t* next,
                             int n_next, int layer, e0_expert_cache c) {
    __shared__ SlotPlan P;
    __shared__ uint32_t prot[E0_MAX_E / 32];
    const int lane = threadIdx.x & 31;
    if (threadIdx.x >= 32) return;
    uint32_t clock = c.counters[0];
    const uint32_t fresh = clock;
    cache_plan_layer(table, occupant, n_slots, E, next, n_next, layer, c, c.scratch, clock, fresh, P, prot, lane);
    if (lane == 0) c.counters[0] = clock;
}

__global__ void k_cache_copy(uint8_t* pool, const uint8_t* bank, e0_expert_cache c, size_t sbytes) {
    const int32_t* plan = c.scratch;
    const int n = plan[0];
    const size_t chunks = sbytes / 16;
    const size_t total = chunks * (size_t)n;
    // four 16-byte loads in flight per thread (the bank may be host memory)
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t q0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q0 < total; q0 += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t q = q0 + u * stride;
            if (q < total) {
                const int i = (int)(q / chunks);
                const int e = plan[4 + 4 * i], src = plan[4 + 4 * i + 2];
                const uint8_t* from = src >= 0 ? c.data + (size_t)src * sbytes : bank + (size_t)e * sbytes;
                v[u] = *reinterpret_cast<const uint4*>(from + (q % chunks) * 16);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t q = q0 + u * stride;
            if (q < total) {
                const int i = (int)(q / chunks);
                const size_t off = (q % chunks) * 16;
                const int s = plan[4 + 4 * i + 1], fill = plan[4 + 4 * i + 3];
                *reinterpret_cast<uint4*>(pool + (size_t)s * sbytes + off) = v[u];
                if (fill >= 0) *reinterpret_cast<uint4*>(c.data + (size_t)fill * sbytes + off) = v[u];
            }
        }
    }
}

// Every layer of a batch planned in order by one warp (one clock, so that no
// copy of the batch evicts an entry another one uses); plans at plans + i *
// CACHE_PLAN_INTS.
__global__ void k_cache_plan_batch(const __grid_constant__ PrefetchBatch B, e0_expert_cache c, int32_t* plans) {
    __shared__ SlotPlan P;
    __shared__ uint32_t prot[E0_MAX_E / 32];
    const int lane = threadIdx.x & 31;
    if (threadIdx.x >= 32) return;
    uint32_t clock = c.counters[0];
    const uint32_t fresh = clock;
    for (int i = 0; i < B.n; ++i) {
        const PrefetchLayer& L = B.l[i];
        cache_plan_layer(L.table, L.occupant, L.n_slots, L.E, L.next, B.K, L.layer, c, plans + (size_t)i * CACHE_PLAN_INTS,
                         clock, fresh, P, prot, lane);
        __syncwarp();
    }
    if (lane == 0) c.counters[0] = clock;
}

// The batch's copies: block group i carries out layer i's plan.
__global__ void k_cache_copy_batch(const __grid_constant__ PrefetchBatch B, e0_expert_cache c, const int32_t* plans) {
    const int li = blockIdx.x / B.per, b = blockIdx.x % B.per;
    const PrefetchLayer& L = B.l[li];
    const int32_t* plan = plans + (size_t)li * CACHE_PLAN_INTS;
    const int n = plan[0];
    const size_t sbytes = B.sbytes, chunks = sbytes / 16;
    const size_t total = chunks * (size_t)n;
    const size_t stride = (size_t)B.per * blockDim.x;
    for (size_t q0 = (size_t)b * blockDim.x + threadIdx.x; q0 < total; q0 += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t q = q0 + u * stride;
            if (q < total) {
                const int i = (int)(q / chunks);
                const int e = plan[4 + 4 * i], src = plan[4 + 4 * i + 2];
                const uint8_t* from = src >= 0 ? c.data + (size_t)src * sbytes : L.bank + (size_t)e * sbytes;
                v[u] = *reinterpret_cast<const uint4*>(from + (q % chunks) * 16);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t q = q0 + u * stride;
            if (q < total) {
                const int i = (int)(q / chunks);
                const size_t off = (q % chunks) * 16;
                const int s2 = plan[4 + 4 * i + 1], fill = plan[4 + 4 * i + 3];
                *reinterpret_cast<uint4*>(L.data + (size_t)s2 * sbytes + off) = v[u];
                if (fill >= 0) *reinterpret_cast<uint4*>(c.data + (size_t)fill * sbytes + off) = v[u];
            }
        }
    }
}

// ================================================================== routing / norm

__global__ void k_route(const float* logits, int T, int E, RouteP rp, int32_t* inds, float* w, uint32_t* st) {
    extern __shared__ float scr[];  // E floats per warp
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x * (blockDim.x >> 5) + warp;
    if (t >= T) return;
    route_warp(logits + (size_t)t * E, E, rp, inds + (size_t)t * rp.K, w + (size_t)t * rp.K, scr + warp * E, st,
               lane);
}

__global__ void k_rmsnorm(const float* r, int H, float eps, float* h) {
    __shared__ float red[32];
    rmsnorm_block(r + (size_t)blockIdx.x * H, h + (size_t)blockIdx.x * H, H, eps, red);
}

// ================================================================== phase kernels

__global__ void __launch_bounds__(PHASE_THREADS) k_router(DecodeArgs A) { phase_router(A, blockIdx.x, gridDim.x); }

__global__ void __launch_bounds__(PHASE_THREADS) k_gateup(DecodeArgs A) {
    extern __shared__ __align__(16) char smem[];
    phase_gateup(A, A.inds, blockIdx.x, gridDim.x, smem);
}

__global__ void __launch_bounds__(PHASE_THREADS) k_down(DecodeArgs A) {
    extern __shared__ __align__(16) char smem[];
    phase_down(A, blockIdx.x, gridDim.x, smem);
}

// ================================================================== stack

struct StackHdr {
    int32_t L, H, I, E, K, hidden, rank;
    RouteP rp;
    int32_t t;
    uint32_t bar_count, bar_gen, bar_abort;
    LayerP* layers;
    int32_t* hist;       // [2][L][K]
    float* wcur;         // [L][K]
    int32_t* pred_inds;  // [2][L][K]
    float* pred_w;       // [2][L][K]
    float* r;            // [H]
    float* h;            // [H]
    float* logits;       // [E]
    float* a;            // [K][I]
    float* gs;           // [I]
    float* us;           // [I]
    float* zg;           // [rank]
    float* zu;           // [rank]
    float* hpre;         // [hidden]
    float* zres;         // [E]
    float* z;            // [E]
    int32_t grid;        // blocks of the persistent kernel
    int32_t smem;        // its dynamic shared memory
    // flag-carrying-word kernel (k_stack_ll): 64-bit (epoch << 32 | fp32) words
    unsigned long long* llR;   // [H] residual stream after each layer
    unsigned long long* llA;   // [(K + 2) I + 2 * 16] a-values, shared pre-activations, LoRA z_g / z_u
    unsigned long long* llLg;  // [E] router logits of a native layer
    unsigned long long* llHp;  // [2][hidden + E] head fc1 outputs and linear-residual outputs, by layer parity
    unsigned long long* llZ;   // [L][E] head logits of each owner
    unsigned long long* llZg;  // [2 * 16] LoRA z_g, z_u of the shared expert
    unsigned long long* llZd;  // [64][16] partial sums of LoRA z_d, one row per CTA holding shared rows
    size_t ll_bytes;           // bytes of the five buffers (cleared by e0_stack_prepare)
    uint32_t ll_abort;         // set when a CTA gave up waiting
    unsigned long long ll_wait_ns;  // a poll gives up after this much device time
    int32_t grid3, smem3, pf_dist, ll_ok;
    int32_t free_sms;  // SMs impl 3 leaves to other streams; the prefetch copies run on that many CTAs
    int32_t* pf_plans;  // [64][4 + 4 E0_MAX_K] plans of a batched prefetch through an expert cache
};

struct TraceP {
    float* r;
    int32_t* inds;
    float* w;
    float* head_logits;
    int32_t* pred_inds;
};

struct WsCarve {
    char* base;
    size_t off;
    template <class T>
    T* take(size_t n) {
        off = (off + 255) & ~(size_t)255;
        T* p = reinterpret_cast<T*>(base + off);
        off += n * sizeof(T);
        return p;
    }
};

static size_t stack_layout(StackHdr* hdr, char* base, int L, int H, int I, int E, int K, int hidden, int rank) {
    WsCarve c{base, 0};
    c.take<StackHdr>(1);
    LayerP* layers = c.take<LayerP>(L);
    int32_t* hist = c.take<int32_t>((size_t)2 * L * K);
    float* wcur = c.take<float>((size_t)L * K);
    int32_t* pi = c.take<int32_t>((size_t)2 * L * K);
    float* pw = c.take<float>((size_t)2 * L * K);
    float* r = c.take<float>(H);
    float* h = c.take<float>(H);
    float* lg = c.take<float>(E);
    float* a = c.take<float>((size_t)K * I);
    float* gs = c.take<float>(I);
    float* us = c.take<float>(I);
    float* zg = c.take<float>(rank > 0 ? rank : 1);
    float* zu = c.take<float>(rank > 0 ? rank : 1);
    float* hp = c.take<float>(hidden > 0 ? hidden : 1);
    float* zr = c.take<float>(E);
    float* z = c.take<float>(E);
    const size_t ll0 = (c.off + 255) & ~(size_t)255;
    unsigned long long* llR = c.take<unsigned long long>(H);
    unsigned long long* llA = c.take<unsigned long long>((size_t)(K + 2) * I + 32);
    unsigned long long* llLg = c.take<unsigned long long>(E);
    unsigned long long* llHp = c.take<unsigned long long>((size_t)2 * ((hidden > 0 ? hidden : 1) + E));
    unsigned long long* llZ = c.take<unsigned long long>((size_t)L * E);
    unsigned long long* llZg = c.take<unsigned long long>(2 * 16);
    unsigned long long* llZd = c.take<unsigned long long>((size_t)64 * 16);
    int32_t* pf_plans = c.take<int32_t>((size_t)PREFETCH_MAX_LAYERS * CACHE_PLAN_INTS);
    if (hdr) {
        hdr->pf_plans = pf_plans;
        hdr->llZg = llZg;
        hdr->llZd = llZd;
        hdr->llR = llR;
        hdr->llA = llA;
        hdr->llLg = llLg;
        hdr->llHp = llHp;
        hdr->llZ = llZ;
        hdr->ll_bytes = c.off - ll0;
        hdr->layers = layers;
        hdr->hist = hist;
        hdr->wcur = wcur;
        hdr->pred_inds = pi;
        hdr->pred_w = pw;
        hdr->r = r;
        hdr->h = h;
        hdr->logits = lg;
        hdr->a = a;
        hdr->gs = gs;
        hdr->us = us;
        hdr->zg = zg;
        hdr->zu = zu;
        hdr->hpre = hp;
        hdr->zres = zr;
        hdr->z = z;
    }
    return c.off + 256;
}

E0_DEV DecodeArgs stack_args(const StackHdr& S, const LayerP& L, const float* h, const float* resid, float* y,
                             const int32_t* inds, const float* w, const int32_t* inds_prev, uint32_t* st) {
    DecodeArgs A;
    A.T = 1;
    A.H = S.H;
    A.I = S.I;
    A.E = S.E;
    A.K = S.K;
    A.x = h;
    A.resid = resid;
    A.inds = inds;
    A.w = w;
    A.inds_prev = inds_prev;
    A.L = L;
    A.a = S.a;
    A.gs = S.gs;
    A.us = S.us;
    A.zg = S.zg;
    A.zu = S.zu;
    A.hpre = S.hpre;
    A.zres = S.zres;
    A.y = y;
    A.z = L.fc1 ? S.z : nullptr;
    A.logits = S.logits;
    A.st = st;
    return A;
}

E0_DEV bool layer_native(const StackHdr& S, const LayerP& L, int t) { return t == 0 || !L.consumer; }

// Route the head logits z of owner layer `l` into the prediction consumed by
// layer l+1 at the next token (one warp).
__device__ __noinline__ void stack_route_head(const StackHdr& S, int l, int t, float* scr, TraceP tr, uint32_t* st, int lane,
                             const float* z = nullptr) {
    if (l + 1 >= S.L) return;
    if (z == nullptr) z = S.z;
    const int np = (t + 1) & 1;
    int32_t* pi = S.pred_inds + ((size_t)np * S.L + (l + 1)) * S.K;
    float* pw = S.pred_w + ((size_t)np * S.L + (l + 1)) * S.K;
    RouteP rp = S.rp;
    rp.logit_bias = nullptr;
    route_warp(z, S.E, rp, pi, pw, scr, st, lane);
    __syncwarp();
    if (tr.head_logits)
        for (int e = lane; e < S.E; e += 32) tr.head_logits[(size_t)l * S.E + e] = __ldcg(z + e);
    if (tr.pred_inds && lane < S.K) tr.pred_inds[(size_t)(l + 1) * S.K + lane] = pi[lane];
}

// Resolve the routing layer l uses at token t into inds/w (one warp).
__device__ __noinline__ void stack_resolve(const StackHdr& S, const LayerP& L, int l, int t, int32_t* inds, float* w, float* scr,
                          uint32_t* st, int lane) {
    if (layer_native(S, L, t)) {
        route_warp(S.logits, S.E, S.rp, inds, w, scr, st, lane);
    } else if (lane < S.K) {
        const size_t o = ((size_t)(t & 1) * S.L + l) * S.K + lane;
        inds[lane] = __ldcg(S.pred_inds + o);
        w[lane] = __ldcg(S.pred_w + o);
    }
    __syncwarp();
}

// ---- chain implementation: one kernel per phase

__global__ void k_stack_norm(StackHdr* Sp, int l, const float* x, TraceP tr) {
    __shared__ float red[32];
    const StackHdr& S = *Sp;
    const float* rin = l == 0 ? x : S.r;
    rmsnorm_block(rin, S.h, S.H, 1e-6f, red);
    if (tr.r)
        for (int j = threadIdx.x; j < S.H; j += blockDim.x) tr.r[(size_t)l * S.H + j] = rin[j];
}

__global__ void __launch_bounds__(PHASE_THREADS) k_stack_router(StackHdr* Sp, int l, uint32_t* st) {
    const StackHdr& S = *Sp;
    const LayerP& L = S.layers[l];
    if (!layer_native(S, L, S.t)) return;
    DecodeArgs A = stack_args(S, L, S.h, nullptr, nullptr, nullptr, nullptr, nullptr, st);
    phase_router(A, blockIdx.x, gridDim.x);
}

__global__ void k_stack_resolve(StackHdr* Sp, int l, TraceP tr, uint32_t* st) {
    extern __shared__ float scr[];
    const StackHdr& S = *Sp;
    const int t = S.t, lane = threadIdx.x & 31;
    int32_t* inds = S.hist + ((size_t)(t & 1) * S.L + l) * S.K;
    float* w = S.wcur + (size_t)l * S.K;
    stack_resolve(S, S.layers[l], l, t, inds, w, scr, st, lane);
    if (lane < S.K) {
        if (tr.inds) tr.inds[(size_t)l * S.K + lane] = inds[lane];
        if (tr.w) tr.w[(size_t)l * S.K + lane] = w[lane];
    }
}

__global__ void __launch_bounds__(PHASE_THREADS) k_stack_gateup(StackHdr* Sp, int l, uint32_t* st) {
    extern __shared__ __align__(16) char smem[];
    const StackHdr& S = *Sp;
    const LayerP& L = S.layers[l];
    const int t = S.t;
    const int32_t* inds = S.hist + ((size_t)(t & 1) * S.L + l) * S.K;
    const int32_t* prev = t > 0 ? S.hist + ((size_t)((t + 1) & 1) * S.L + l) * S.K : nullptr;
    DecodeArgs A = stack_args(S, L, S.h, nullptr, nullptr, inds, S.wcur + (size_t)l * S.K, prev, st);
    phase_gateup(A, inds, blockIdx.x, gridDim.x, smem);
}

__global__ void __launch_bounds__(PHASE_THREADS) k_stack_down(StackHdr* Sp, int l, const float* x, float* r_out,
                                                              uint32_t* st) {
    extern __shared__ __align__(16) char smem[];
    const StackHdr& S = *Sp;
    const LayerP& L = S.layers[l];
    const int t = S.t;
    const int32_t* inds = S.hist + ((size_t)(t & 1) * S.L + l) * S.K;
    const float* rin = l == 0 ? x : S.r;
    float* y = l == S.L - 1 ? r_out : S.r;
    DecodeArgs A = stack_args(S, L, S.h, rin, y, inds, S.wcur + (size_t)l * S.K, nullptr, st);
    phase_down(A, blockIdx.x, gridDim.x, smem);
}

__global__ void k_stack_head(StackHdr* Sp, int l, TraceP tr, uint32_t* st) {
    extern __shared__ float scr[];
    const StackHdr& S = *Sp;
    if (!S.layers[l].fc1) return;
    stack_route_head(S, l, S.t, scr, tr, st, threadIdx.x & 31);
}

__global__ void k_stack_finish(StackHdr* Sp, const float* r_out, TraceP tr) {
    StackHdr& S = *Sp;
    if (tr.r)
        for (int j = threadIdx.x; j < S.H; j += blockDim.x) tr.r[(size_t)S.L * S.H + j] = r_out[j];
    __syncthreads();
    if (threadIdx.x == 0) S.t = S.t + 1;
}

// ---- persistent implementation: the whole token in one cooperative kernel

E0_DEV void grid_barrier(StackHdr* S, uint32_t* st) {
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned gen;
        asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(gen) : "l"(&S->bar_gen) : "memory");
        __threadfence();
        const unsigned arrived = atomicAdd(&S->bar_count, 1u);
        if (arrived == gridDim.x - 1) {
            atomicExch(&S->bar_count, 0u);
            __threadfence();
            asm volatile("st.release.gpu.u32 [%0], %1;" ::"l"(&S->bar_gen), "r"(gen + 1) : "memory");
        } else {
            uint32_t it = 0;
            while (true) {
                unsigned cur, ab;
                asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(cur) : "l"(&S->bar_gen) : "memory");
                if (cur != gen) break;
                asm volatile("ld.relaxed.gpu.u32 %0, [%1];" : "=r"(ab) : "l"(&S->bar_abort) : "memory");
                if (ab) break;
                if (++it > BARRIER_SPIN_LIMIT) {
                    set_status(st, E0_ST_TIMEOUT);
                    atomicExch(&S->bar_abort, 1u);
                    break;
                }
                if (it > 64) __nanosleep(32);
            }
        }
        __threadfence();
    }
    __syncthreads();
}

struct PersistSmem {
    size_t h, inds, w, scr, red, phase, total;
    __host__ __device__ PersistSmem(int H, int E, int K, size_t phase_bytes) {
        h = 0;
        inds = h + (size_t)H * 4;
        w = inds + 128;
        scr = w + 128;
        red = scr + (size_t)2 * E * 4;
        phase = red + 128;
        phase = (phase + 15) & ~(size_t)15;
        total = phase + phase_bytes;
        (void)K;
    }
};

__global__ void __launch_bounds__(PHASE_THREADS) k_stack_token(StackHdr* Sp, const float* x, float* r_out, TraceP tr,
                                                               uint32_t* st) {
    extern __shared__ __align__(16) char smem[];
    StackHdr& S = *Sp;
    const int t = S.t;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t phase_bytes = (size_t)S.smem;
    const PersistSmem lay(S.H, S.E, S.K, 0);
    float* hbuf = reinterpret_cast<float*>(smem + lay.h);
    int32_t* inds_s = reinterpret_cast<int32_t*>(smem + lay.inds);
    float* w_s = reinterpret_cast<float*>(smem + lay.w);
    float* scr = reinterpret_cast<float*>(smem + lay.scr);
    float* red = reinterpret_cast<float*>(smem + lay.red);
    char* psm = smem + lay.phase;
    (void)phase_bytes;

    for (int l = 0; l < S.L; ++l) {
        const LayerP L = S.layers[l];
        const bool native = layer_native(S, L, t);
        const float* rin = l == 0 ? x : S.r;
        // every block normalises the residual stream itself
        {
            float s = 0.f;
            for (int j = threadIdx.x; j < S.H; j += blockDim.x) {
                const float v = __ldcg(rin + j);
                hbuf[j] = v;
                s = fmaf(v, v, s);
            }
            s = warp_sum(s);
            if (lane == 0) red[warp] = s;
            __syncthreads();
            if (warp == 0) {
                float v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.f;
                v = warp_sum(v);
                if (lane == 0) red[0] = v;
            }
            __syncthreads();
            const float denom = sqrtf(red[0] / (float)S.H + 1e-6f);
            if (blockIdx.x == 0 && tr.r)
                for (int j = threadIdx.x; j < S.H; j += blockDim.x) tr.r[(size_t)l * S.H + j] = hbuf[j];
            __syncthreads();
            for (int j = threadIdx.x; j < S.H; j += blockDim.x) hbuf[j] = hbuf[j] / denom;
            __syncthreads();
        }
        if (native) {
            DecodeArgs A = stack_args(S, L, hbuf, nullptr, nullptr, nullptr, nullptr, nullptr, st);
            phase_router(A, blockIdx.x, gridDim.x);
            grid_barrier(Sp, st);
        }
        // routing of this layer (every block, warp 0) and the previous owner's prediction (block 0, warp 1)
        if (warp == 0) {
            stack_resolve(S, L, l, t, inds_s, w_s, scr, blockIdx.x == 0 ? st : nullptr, lane);
            if (blockIdx.x == 0 && lane < S.K) {
                const size_t o = ((size_t)(t & 1) * S.L + l) * S.K + lane;
                S.hist[o] = inds_s[lane];
                S.wcur[(size_t)l * S.K + lane] = w_s[lane];
                if (tr.inds) tr.inds[(size_t)l * S.K + lane] = inds_s[lane];
                if (tr.w) tr.w[(size_t)l * S.K + lane] = w_s[lane];
            }
        } else if (warp == 1 && blockIdx.x == 0 && l > 0 && S.layers[l - 1].fc1) {
            stack_route_head(S, l - 1, t, scr + S.E, tr, st, lane);
        }
        __syncthreads();
        {
            const int32_t* prev = t > 0 ? S.hist + ((size_t)((t + 1) & 1) * S.L + l) * S.K : nullptr;
            DecodeArgs A = stack_args(S, L, hbuf, nullptr, nullptr, inds_s, w_s, prev, st);
            phase_gateup(A, inds_s, blockIdx.x, gridDim.x, psm);
        }
        grid_barrier(Sp, st);
        {
            const int32_t* inds = S.hist + ((size_t)(t & 1) * S.L + l) * S.K;
            float* y = l == S.L - 1 ? r_out : S.r;
            DecodeArgs A = stack_args(S, L, hbuf, rin, y, inds, S.wcur + (size_t)l * S.K, nullptr, st);
            phase_down(A, blockIdx.x, gridDim.x, psm);
        }
        grid_barrier(Sp, st);
    }
    if (blockIdx.x == 0) {
        if (warp == 1 && S.layers[S.L - 1].fc1) stack_route_head(S, S.L - 1, t, scr + S.E, tr, st, lane);
        if (tr.r)
            for (int j = threadIdx.x; j < S.H; j += blockDim.x) tr.r[(size_t)S.L * S.H + j] = __ldcg(r_out + j);
        __syncthreads();
        if (threadIdx.x == 0) S.t = t + 1;
    }
}

#include "e0_stack_ll.cuh"

// Layer shapes the flag-carrying-word kernel is built for (other shapes: impl 0).
using LLS35K4 = LLShape<2048, 512, 256, 4>;
using LLS35K2 = LLShape<2048, 512, 256, 2>;
using LLS35K8 = LLShape<2048, 512, 256, 8>;
using LLS8B = LLShape<1536, 384, 128, 8>;
using LLSTiny = LLShape<256, 128, 16, 4>;

static const void* ll_kernel(int H, int I, int E, int K) {
    if (H == 2048 && I == 512 && E == 256) {
        if (K == 4) return (const void*)k_stack_ll<LLS35K4>;
        if (K == 2) return (const void*)k_stack_ll<LLS35K2>;
        if (K == 8) return (const void*)k_stack_ll<LLS35K8>;
    }
    if (H == 1536 && I == 384 && E == 128 && K == 8) return (const void*)k_stack_ll<LLS8B>;
    if (H == 256 && I == 128 && E == 16 && K == 4) return (const void*)k_stack_ll<LLSTiny>;
    return nullptr;
}

// ================================================================== host side

static int g_num_sms = 0;
static int g_smem_optin = 0;
static std::once_flag g_init;

static void init_attrs() {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    const int big = 200 * 1024;
    cudaFuncSetAttribute(k_gateup, cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    cudaFuncSetAttribute(k_down, cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    cudaFuncSetAttribute(k_stack_gateup, cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    cudaFuncSetAttribute(k_stack_down, cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    cudaFuncSetAttribute(k_stack_token, cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    cudaDeviceGetAttribute(&g_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (g_smem_optin <= 0) g_smem_optin = big;
    for (const void* f : {(const void*)k_stack_ll<LLS35K4>, (const void*)k_stack_ll<LLS35K2>,
                          (const void*)k_stack_ll<LLS35K8>, (const void*)k_stack_ll<LLS8B>, (const void*)k_stack_ll<LLSTiny>})
        cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, g_smem_optin);
}

// largest dynamic shared memory one block may take
static size_t smem_optin() {
    num_sms();
    return (size_t)g_smem_optin;
}

int num_sms() {
    std::call_once(g_init, init_attrs);
    return g_num_sms > 0 ? g_num_sms : 148;
}

static int phase_grid(long warps) {
    long blocks = (warps + (PHASE_THREADS / 32) - 1) / (PHASE_THREADS / 32);
    const long cap = (long)num_sms() * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return (int)blocks;
}

static RouteP to_route(const e0_route_params* rp) {
    RouteP r;
    r.mode = rp->mode;
    r.K = rp->K;
    r.n_groups = rp->n_groups > 0 ? rp->n_groups : 1;
    r.topk_groups = rp->topk_groups > 0 ? rp->topk_groups : 1;
    r.scale = rp->scale;
    r.logit_bias = rp->logit_bias;
    return r;
}

static LayerP to_layer(const e0_slot_pool* pool, const uint16_t* W_r, const e0_shared_expert* sh,
                       const e0_prerouter* head, int consumer) {
    LayerP L;
    memset(&L, 0, sizeof(L));
    if (pool) {
        L.pool = pool->data;
        L.table = pool->slot_table;
        L.n_slots = pool->n_slots;
    }
    L.W_r = reinterpret_cast<const __half*>(W_r);
    if (sh) {
        L.sh = sh->data;
        if (sh->A_gate) {
            L.Ag = reinterpret_cast<const __half*>(sh->A_gate);
            L.Bg = reinterpret_cast<const __half*>(sh->B_gate);
            L.Au = reinterpret_cast<const __half*>(sh->A_up);
            L.Bu = reinterpret_cast<const __half*>(sh->B_up);
            L.Ad = reinterpret_cast<const __half*>(sh->A_down);
            L.Bd = reinterpret_cast<const __half*>(sh->B_down);
            L.rank = sh->rank;
            L.lscale = sh->alpha / (float)sh->rank;
        }
    }
    if (head) {
        L.fc1 = reinterpret_cast<const __half*>(head->fc1);
        L.b1 = reinterpret_cast<const __half*>(head->b1);
        L.fc2 = reinterpret_cast<const __half*>(head->fc2);
        L.b2 = reinterpret_cast<const __half*>(head->b2);
        L.lres = reinterpret_cast<const __half*>(head->lres);
        L.hidden = head->hidden;
    }
    L.consumer = consumer;
    return L;
}

static inline int cuda_ok(cudaError_t e) { return e == cudaSuccess ? E0_OK : E0_ERR_CUDA; }
static inline int launch_ok() { return cuda_ok(cudaGetLastError()); }

// ---- packing

int pack_experts(const e0_expert_q* src, int n, const e0_slot_pool* dst, const int32_t* dst_slots,
                 const int32_t* expert_ids, cudaStream_t s) {
    num_sms();
    const size_t sb = slot_bytes(dst->H, dst->I);
    for (int i = 0; i < n; ++i) {
        uint8_t* d = dst->data + (size_t)dst_slots[i] * sb;
        k_pack_expert<<<num_sms() * 2, 256, 0, s>>>(src[i], d, dst->H, dst->I, dst->slot_table, dst->occupant,
                                                     expert_ids ? expert_ids[i] : -1, dst_slots[i]);
        if (launch_ok() != E0_OK) return E0_ERR_CUDA;
    }
    return cuda_ok(cudaStreamSynchronize(s));
}

int slot_update(const e0_slot_pool* p, const int32_t* next, int n_next, const int32_t* cur, int n_cur,
                const uint8_t* bank, uint32_t* st, cudaStream_t s, int grid) {
    const size_t sb = slot_bytes(p->H, p->I);
    k_slot_copy<<<grid > 0 ? grid : num_sms(), 512, 0, s>>>(p->slot_table, p->occupant, p->data, p->n_slots, p->E, next, n_next, cur,
                                          n_cur, bank, sb);
    if (launch_ok() != E0_OK) return E0_ERR_CUDA;
    k_slot_commit<<<1, 32, 0, s>>>(p->slot_table, p->occupant, p->n_slots, p->E, next, n_next, cur, n_cur, st);
    return launch_ok();
}

int route(const float* logits, int T, int E, const e0_route_params* rp, int32_t* inds, float* w, uint32_t* st,
          cudaStream_t s) {
    if (T == 0) return E0_OK;
    const int wpb = 4;
    k_route<<<(T + wpb - 1) / wpb, 32 * wpb, (size_t)wpb * E * sizeof(float), s>>>(logits, T, E, to_route(rp), inds,
                                                                                   w, st);
    return launch_ok();
}

int rmsnorm(const float* r, int T, int H, float eps, float* h, cudaStream_t s) {
    if (T == 0) return E0_OK;
    k_rmsnorm<<<T, 256, 0, s>>>(r, H, eps, h);
    return launch_ok();
}

// ---- MoE block

struct BlockWs {
    float* logits;
    int32_t* inds;
    float* w;
    float* a;
    float* gs;
    float* us;
    float* zg;
    float* zu;
    float* hpre;
    float* zres;
    size_t bytes;
};

static BlockWs block_ws(char* base, int T, int H, int I, int E, int K, int rank, int hidden) {
    const int Tc = T < 8 ? T : 8;
    WsCarve c{base, 0};
    BlockWs b;
    b.logits = c.take<float>((size_t)T * E);
    b.inds = c.take<int32_t>((size_t)T * K);
    b.w = c.take<float>((size_t)T * K);
    b.a = c.take<float>((size_t)Tc * K * I);
    b.gs = c.take<float>((size_t)Tc * I);
    b.us = c.take<float>((size_t)Tc * I);
    b.zg = c.take<float>((size_t)Tc * (rank > 0 ? rank : 1));
    b.zu = c.take<float>((size_t)Tc * (rank > 0 ? rank : 1));
    b.hpre = c.take<float>((size_t)Tc * (hidden > 0 ? hidden : 1));
    b.zres = c.take<float>((size_t)T * E);
    b.bytes = c.off + 256;
    (void)H;
    return b;
}

size_t block_ws_bytes(int T, int H, int I, int E, int K, int rank, int hidden) {
    return block_ws(nullptr, T, H, I, E, K, rank, hidden).bytes;
}

int moe_block_forward(const float* x, int T, const e0_slot_pool* pool, const uint16_t* W_r,
                      const e0_route_params* rp, const int32_t* inds_in, const float* w_in,
                      const e0_shared_expert* sh, float* y, int32_t* inds_out, float* w_out, void* ws,
                      uint32_t* st, cudaStream_t s) {
    num_sms();
    const int H = pool->H, I = pool->I, E = pool->E, K = rp->K;
    const int rank = (sh && sh->A_gate) ? sh->rank : 0;
    BlockWs b = block_ws(reinterpret_cast<char*>(ws), T, H, I, E, K, 64, 0);
    LayerP L = to_layer(pool, W_r, sh, nullptr, 0);
    const int32_t* inds = inds_in;
    const float* w = w_in;
    if (!inds_in) {
        DecodeArgs A;
        memset(&A, 0, sizeof(A));
        A.T = T;
        A.H = H;
        A.I = I;
        A.E = E;
        A.K = K;
        A.x = x;
        A.L = L;
        A.logits = b.logits;
        A.st = st;
        const int R = (H / GROUP) >= 32 ? 1 : 32 / (H / GROUP);
        const long warps = (long)T * ((E + R - 1) / R);
        k_router<<<phase_grid(warps), PHASE_THREADS, 0, s>>>(A);
        if (launch_ok() != E0_OK) return E0_ERR_CUDA;
        int32_t* io = inds_out ? inds_out : b.inds;
        float* wo = w_out ? w_out : b.w;
        int rc = route(b.logits, T, E, rp, io, wo, st, s);
        if (rc) return rc;
        inds = io;
        w = wo;
    } else {
        if (inds_out && inds_out != inds_in &&
            cudaMemcpyAsync(inds_out, inds_in, (size_t)T * K * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return E0_ERR_CUDA;
        if (w_out && w_out != w_in &&
            cudaMemcpyAsync(w_out, w_in, (size_t)T * K * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return E0_ERR_CUDA;
    }
    for (int t0 = 0; t0 < T; t0 += 8) {
        const int Tc = T - t0 < 8 ? T - t0 : 8;
        DecodeArgs A;
        memset(&A, 0, sizeof(A));
        A.T = Tc;
        A.H = H;
        A.I = I;
        A.E = E;
        A.K = K;
        A.x = x + (size_t)t0 * H;
        A.resid = nullptr;
        A.inds = inds + (size_t)t0 * K;
        A.w = w + (size_t)t0 * K;
        A.L = L;
        A.a = b.a;
        A.gs = b.gs;
        A.us = b.us;
        A.zg = b.zg;
        A.zu = b.zu;
        A.hpre = b.hpre;
        A.zres = b.zres;
        A.y = y + (size_t)t0 * H;
        A.st = st;
        const int R = (H / GROUP) >= 32 ? 1 : 32 / (H / GROUP);
        long warps = (long)Tc * (K + 1) * ((I + R - 1) / R) + 2 * rank;
        const GateUpSmem gsm(Tc, H, K);
        k_gateup<<<phase_grid(warps), PHASE_THREADS, gsm.total, s>>>(A);
        if (launch_ok() != E0_OK) return E0_ERR_CUDA;
        const int RI = (I / GROUP) >= 32 ? 1 : 32 / (I / GROUP);
        warps = (long)Tc * ((H + RI - 1) / RI);
        const DownSmem dsm(Tc, I, K, sh != nullptr, rank, 0);
        k_down<<<phase_grid(warps), PHASE_THREADS, dsm.total, s>>>(A);
        if (launch_ok() != E0_OK) return E0_ERR_CUDA;
    }
    return E0_OK;
}

// ---- prerouter head

size_t head_ws_bytes(int T, int H, int hidden, int E, int K) {
    WsCarve c{nullptr, 0};
    c.take<float>((size_t)T * hidden);
    c.take<float>((size_t)T * E);
    c.take<float>((size_t)T * E);
    (void)H;
    (void)K;
    return c.off + 256;
}

int prerouter_forward(const float* h, int T, const int32_t* inds_cur, const int32_t* inds_prev,
                      const e0_prerouter* head, const e0_route_params* rp, float* logits_out, int32_t* inds_next,
                      float* w_next, void* ws, uint32_t* st, cudaStream_t s) {
    num_sms();
    const int H = head->H, E = head->E, K = rp->K, hidden = head->hidden;
    WsCarve c{reinterpret_cast<char*>(ws), 0};
    float* hpre = c.take<float>((size_t)T * hidden);
    float* zres = c.take<float>((size_t)T * E);
    float* zbuf = c.take<float>((size_t)T * E);
    float* z = logits_out ? logits_out : zbuf;
    LayerP L = to_layer(nullptr, nullptr, nullptr, head, 0);
    for (int t0 = 0; t0 < T; t0 += 8) {
        const int Tc = T - t0 < 8 ? T - t0 : 8;
        DecodeArgs A;
        memset(&A, 0, sizeof(A));
        A.T = Tc;
        A.H = H;
        A.I = GROUP;
        A.E = E;
        A.K = K;
        A.x = h + (size_t)t0 * H;
        A.inds = inds_cur + (size_t)t0 * K;
        A.inds_prev = inds_prev ? inds_prev + (size_t)t0 * K : nullptr;
        A.L = L;
        A.hpre = hpre + (size_t)t0 * hidden;
        A.zres = zres + (size_t)t0 * E;
        A.z = z + (size_t)t0 * E;
        A.st = st;
        const int R = (H / GROUP) >= 32 ? 1 : 32 / (H / GROUP);
        long warps = (long)Tc * ((hidden + E + R - 1) / R);
        const GateUpSmem gsm(Tc, H, K);
        k_gateup<<<phase_grid(warps), PHASE_THREADS, gsm.total, s>>>(A);
        if (launch_ok() != E0_OK) return E0_ERR_CUDA;
        const int Rh = (hidden / GROUP) >= 32 ? 1 : 32 / (hidden / GROUP);
        warps = (long)Tc * ((E + Rh - 1) / Rh);
        const DownSmem dsm(Tc, GROUP, 0, false, 0, hidden);
        k_down<<<phase_grid(warps), PHASE_THREADS, dsm.total, s>>>(A);
        if (launch_ok() != E0_OK) return E0_ERR_CUDA;
    }
    e0_route_params hr = *rp;
    hr.logit_bias = nullptr;
    return route(z, T, E, &hr, inds_next, w_next, st, s);
}

// ---- stack

size_t stack_ws_bytes(int L, int H, int I, int E, int K, int hidden) {
    return stack_layout(nullptr, nullptr, L, H, I, E, K, hidden, E0_MAX_LORA_RANK);
}

// Host copies of every prepared stack header, keyed by workspace address, so
// that a step needs no device read-back (and can be captured in a graph).
static std::mutex g_stack_mu;
static std::map<const void*, StackHdr> g_stacks;

// Geometry of the flag-carrying-word kernel: one CTA per SM, and whether every
// layer's work split fits the kernel's per-CTA limits (ll_ok = 0: impl 3
// returns E0_ERR_UNSUPPORTED for this stack).
static void ll_geometry(StackHdr* hdr, const e0_stack_layer* layers, int L, int H, int I, int E, int K) {
    // SMs left free for kernels on other streams (the host-tier copies of a
    // streamed stack): a cooperative launch cannot start until every one of its
    // CTAs is resident, so a grid over all SMs waits out any running copy kernel
    int free_sms = 0;
    if (const char* env = getenv("E0MOE_LL_FREE_SMS")) {
        const int v = atoi(env);
        if (v >= 0 && v <= 64) free_sms = v;
    }
    const int nb = num_sms() - free_sms > 1 ? num_sms() - free_sms : 1;
    hdr->grid3 = nb;
    hdr->free_sms = free_sms;
    hdr->pf_dist = LL_PF_DIST;
    if (const char* env = getenv("E0MOE_PF_DIST")) {
        const int v = atoi(env);
        if (v >= 0 && v <= 64) hdr->pf_dist = v;
    }
    hdr->ll_wait_ns = LL_WAIT_NS;
    if (const char* env = getenv("E0MOE_WAIT_US")) {
        const long v = atol(env);
        if (v >= 1 && v <= 10000000) hdr->ll_wait_ns = (unsigned long long)v * 1000ull;
    }
    int hidden = 0;
    for (int l = 0; l < L; ++l)
        if (layers[l].head && layers[l].head->hidden > hidden) hidden = layers[l].head->hidden;
    const LLSmem lay(H, I, E, L, K, hidden, nb);
    const LLGeo geo(H, I, E, K, hidden, nb);
    hdr->smem3 = (int32_t)lay.total;
    const void* fn = ll_kernel(H, I, E, K);
    bool ok = fn != nullptr && (H + 2 * E) % 8 == 0 &&
              (size_t)lay.total <= smem_optin() && geo.nr <= LL_MAXROWS && (K + 1) * I / 32 <= LL_NW * LL_MAXQ;
    const int GH = H / GROUP, R = GH >= 32 ? 1 : 32 / GH;
    auto cdiv = [](long a, long b) { return (int)((a + b - 1) / b); };
    auto al16 = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
    for (int l = 0; l < L && ok; ++l) {
        const e0_stack_layer& ly = layers[l];
        const bool sh = ly.shared != nullptr;
        const bool lora = sh && ly.shared->A_gate != nullptr;
        const int nk = K + (sh ? 1 : 0);
        if (cdiv((long)nk * I, nb) > LL_NW * LL_MAXA * R) ok = false;
        if (!al16(ly.pool.data) || !al16(ly.W_router) || (sh && !al16(ly.shared->data))) ok = false;
        if (lora) {
            const e0_shared_expert* x = ly.shared;
            if (x->rank % 8 != 0 || x->rank > LL_RANK || nb < 2 * x->rank || cdiv((long)nk * I, nb) > 32) ok = false;
            if (!al16(x->A_gate) || !al16(x->A_up) || !al16(x->B_gate) || !al16(x->B_up) || !al16(x->B_down)) ok = false;
            // CTAs holding shared-expert rows
            int s0 = 0;
            while (s0 < nb && (int)((long)nk * I * (s0 + 1) / nb) <= K * I) ++s0;
            if (nb - s0 > LL_MAX_SHCTA) ok = false;
        }
        if (ly.head && l + 1 < L) {
            const int rows = cdiv((long)ly.head->hidden + E, nb);
            if (ly.head->hidden % 256 != 0 || rows > LL_MAXROWS || rows * (H / 256) > LL_NW * LL_MAXB1) ok = false;
            if (!al16(ly.head->fc1) || !al16(ly.head->lres) || !al16(ly.head->fc2)) ok = false;
        }
        if (l >= 1 && layers[l - 1].head && cdiv(E, nb) * (layers[l - 1].head->hidden / 256) > LL_NW) ok = false;
        if (cdiv(E, nb) * (H / 256) > LL_MAX_RITEMS) ok = false;
    }
    int per_sm = 0;
    if (ok && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, LL_THREADS, lay.total) != cudaSuccess) {
        cudaGetLastError();
        per_sm = 0;
    }
    hdr->ll_ok = ok && per_sm >= 1 ? 1 : 0;
}

int stack_prepare(const e0_stack_layer* layers, int L, int H, int I, int E, const e0_route_params* rp, void* ws,
                  cudaStream_t s) {
    num_sms();
    int hidden = 0, rank = 0;
    for (int l = 0; l < L; ++l) {
        if (layers[l].head && layers[l].head->hidden > hidden) hidden = layers[l].head->hidden;
        if (layers[l].shared && layers[l].shared->A_gate && layers[l].shared->rank > rank) rank = layers[l].shared->rank;
    }
    StackHdr hdr;
    memset(&hdr, 0, sizeof(hdr));
    stack_layout(&hdr, reinterpret_cast<char*>(ws), L, H, I, E, rp->K, hidden, E0_MAX_LORA_RANK);
    hdr.L = L;
    hdr.H = H;
    hdr.I = I;
    hdr.E = E;
    hdr.K = rp->K;
    hdr.hidden = hidden;
    hdr.rank = rank;
    hdr.rp = to_route(rp);
    hdr.t = 0;
    // persistent kernel geometry
    const size_t gs = GateUpSmem(1, H, rp->K).total;
    const size_t ds = DownSmem(1, I, rp->K, true, E0_MAX_LORA_RANK, hidden > 0 ? hidden : GROUP).total;
    const size_t ps = gs > ds ? gs : ds;
    const PersistSmem lay(H, E, rp->K, ps);
    hdr.smem = (int32_t)ps;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_stack_token, PHASE_THREADS, lay.total);
    if (per_sm < 1) per_sm = 1;
    if (per_sm > 2) per_sm = 2;
    hdr.grid = num_sms() * per_sm;
    ll_geometry(&hdr, layers, L, H, I, E, rp->K);
    LayerP* hl = new LayerP[L];
    for (int l = 0; l < L; ++l)
        hl[l] = to_layer(&layers[l].pool, layers[l].W_router, layers[l].shared, layers[l].head, layers[l].consumer);
    int rc = E0_OK;
    if (cudaMemcpyAsync(ws, &hdr, sizeof(hdr), cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(hdr.layers, hl, sizeof(LayerP) * L, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemsetAsync(hdr.hist, 0xff, sizeof(int32_t) * 2 * L * rp->K, s) != cudaSuccess ||
        cudaMemsetAsync(hdr.llR, 0, hdr.ll_bytes, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        rc = E0_ERR_CUDA;
    delete[] hl;
    if (rc == E0_OK) {
        std::lock_guard<std::mutex> g(g_stack_mu);
        g_stacks[ws] = hdr;
    }
    return rc;
}

bool stack_known(const void* ws) {
    std::lock_guard<std::mutex> g(g_stack_mu);
    return g_stacks.count(ws) != 0;
}

static TraceP trace_of(const e0_stack_trace* trace) {
    TraceP tr;
    memset(&tr, 0, sizeof(tr));
    if (trace) {
        tr.r = trace->r;
        tr.inds = trace->inds;
        tr.w = trace->w;
        tr.head_logits = trace->head_logits;
        tr.pred_inds = trace->pred_inds;
    }
    return tr;
}

static bool stack_hdr(const void* ws, StackHdr* out) {
    std::lock_guard<std::mutex> g(g_stack_mu);
    auto it = g_stacks.find(ws);
    if (it == g_stacks.end()) return false;
    *out = it->second;
    return true;
}

// Layers [lb, le) of the current token with the flag-carrying-word kernel:
// one cooperative launch (its CTAs wait on words the others write, so they
// must be resident together; a launch that cannot guarantee it is an error).
static int stack_step_ll(const float* x, float* r_out, void* ws, const StackHdr& hdr, int lb, int le,
                         const e0_stack_trace* trace, uint32_t* st, cudaStream_t s) {
    if (!hdr.ll_ok) return E0_ERR_UNSUPPORTED;
    StackHdr* Sp = reinterpret_cast<StackHdr*>(ws);
    TraceP tr = trace_of(trace);
    void* args[] = {&Sp, (void*)&x, &r_out, &tr, &st, &lb, &le};
    const void* fn = ll_kernel(hdr.H, hdr.I, hdr.E, hdr.K);
    if (!fn) return E0_ERR_UNSUPPORTED;
    return cuda_ok(cudaLaunchCooperativeKernel(fn, dim3(hdr.grid3), dim3(LL_THREADS), args, (size_t)hdr.smem3, s));
}

// Layers [lb, le) of the current token (the flag-carrying-word kernel).
int stack_step_range(const float* x, float* r_out, void* ws, int lb, int le, const e0_stack_trace* trace, uint32_t* st,
                     cudaStream_t s) {
    num_sms();
    StackHdr hdr;
    if (!stack_hdr(ws, &hdr)) return E0_ERR_ARG;
    if (lb < 0 || le > hdr.L || lb >= le) return E0_ERR_ARG;
    if (le == hdr.L && !r_out) return E0_ERR_NULL;
    if (lb == 0 && !x) return E0_ERR_NULL;
    return stack_step_ll(x, r_out, ws, hdr, lb, le, trace, st, s);
}

// New layer descriptors for a prepared stack, keeping its routing history,
// predictions and token counter; the layers' configuration must not change.
int stack_update_layers(void* ws, const e0_stack_layer* layers, int L, cudaStream_t s) {
    StackHdr hdr;
    if (!stack_hdr(ws, &hdr)) return E0_ERR_ARG;
    if (L != hdr.L) return E0_ERR_ARG;
    LayerP* hl = new LayerP[L];
    LayerP* cur = new LayerP[L];
    int rc = E0_OK;
    if (cudaMemcpyAsync(cur, hdr.layers, sizeof(LayerP) * L, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        rc = E0_ERR_CUDA;
    for (int l = 0; l < L && rc == E0_OK; ++l) {
        hl[l] = to_layer(&layers[l].pool, layers[l].W_router, layers[l].shared, layers[l].head, layers[l].consumer);
        const bool same = (hl[l].sh != nullptr) == (cur[l].sh != nullptr) && (hl[l].Ag != nullptr) == (cur[l].Ag != nullptr) &&
                          hl[l].rank == cur[l].rank && (hl[l].fc1 != nullptr) == (cur[l].fc1 != nullptr) &&
                          hl[l].hidden == cur[l].hidden && hl[l].consumer == cur[l].consumer;
        if (!same) rc = E0_ERR_ARG;
    }
    if (rc == E0_OK && (cudaMemcpyAsync(hdr.layers, hl, sizeof(LayerP) * L, cudaMemcpyHostToDevice, s) != cudaSuccess ||
                        cudaStreamSynchronize(s) != cudaSuccess))
        rc = E0_ERR_CUDA;
    delete[] hl;
    delete[] cur;
    return rc;
}

// Bring the experts predicted for token t_next of `layer` into `pool`.
int stack_prefetch_experts(void* ws, int layer, int t_next, const e0_slot_pool* pool, const uint8_t* bank, uint32_t* st,
                           cudaStream_t s) {
    StackHdr hdr;
    if (!stack_hdr(ws, &hdr)) return E0_ERR_ARG;
    if (layer < 0 || layer >= hdr.L || t_next < 1) return E0_ERR_ARG;
    const int32_t* next = hdr.pred_inds + ((size_t)(t_next & 1) * hdr.L + layer) * hdr.K;
    return slot_update(pool, next, hdr.K, nullptr, 0, bank, st, s, hdr.free_sms);
}

int stack_prefetch_experts_batch(void* ws, const int32_t* layers, int n, int t_next, const e0_slot_pool* pools,
                                 const uint8_t* const* banks, uint32_t* st, cudaStream_t s) {
    StackHdr hdr;
    if (!stack_hdr(ws, &hdr)) return E0_ERR_ARG;
    if (n < 0 || n > PREFETCH_MAX_LAYERS || t_next < 1) return E0_ERR_ARG;
    if (n == 0) return E0_OK;
    PrefetchBatch B;
    memset(&B, 0, sizeof(B));
    B.n = n;
    B.K = hdr.K;
    for (int i = 0; i < n; ++i) {
        const int layer = layers[i];
        if (layer < 0 || layer >= hdr.L) return E0_ERR_ARG;
        if (pools[i].H != pools[0].H || pools[i].I != pools[0].I) return E0_ERR_ARG;
        PrefetchLayer& L = B.l[i];
        L.table = pools[i].slot_table;
        L.occupant = pools[i].occupant;
        L.data = pools[i].data;
        L.bank = banks[i];
        L.next = hdr.pred_inds + ((size_t)(t_next & 1) * hdr.L + layer) * hdr.K;
        L.n_slots = pools[i].n_slots;
        L.E = pools[i].E;
        L.layer = layer;
    }
    B.sbytes = slot_bytes(pools[0].H, pools[0].I);
    // four 512-thread blocks per SM the copies may use, shared out over the layers
    const int blocks = (hdr.free_sms > 0 ? hdr.free_sms : num_sms()) * 4;
    B.per = blocks / n > 1 ? blocks / n : 1;
    k_slot_copy_batch<<<n * B.per, 512, 0, s>>>(B);
    if (launch_ok() != E0_OK) return E0_ERR_CUDA;
    k_slot_commit_batch<<<n, 32, 0, s>>>(B, st);
    return launch_ok();
}

int stack_prefetch_experts_cached_batch(void* ws, const int32_t* layers, int n, int t_next, const e0_slot_pool* pools,
                                        const uint8_t* const* banks, const e0_expert_cache* c, uint32_t* st,
                                        cudaStream_t s) {
    StackHdr hdr;
    if (!stack_hdr(ws, &hdr)) return E0_ERR_ARG;
    if (n < 0 || n > PREFETCH_MAX_LAYERS || t_next < 1) return E0_ERR_ARG;
    if (n == 0) return E0_OK;
    PrefetchBatch B;
    memset(&B, 0, sizeof(B));
    B.n = n;
    B.K = hdr.K;
    for (int i = 0; i < n; ++i) {
        const int layer = layers[i];
        if (layer < 0 || layer >= hdr.L) return E0_ERR_ARG;
        if (pools[i].H != pools[0].H || pools[i].I != pools[0].I) return E0_ERR_ARG;
        if ((long)(layer + 1) * pools[i].E > c->n_keys) return E0_ERR_ARG;
        PrefetchLayer& L = B.l[i];
        L.table = pools[i].slot_table;
        L.occupant = pools[i].occupant;
        L.data = pools[i].data;
        L.bank = banks[i];
        L.next = hdr.pred_inds + ((size_t)(t_next & 1) * hdr.L + layer) * hdr.K;
        L.n_slots = pools[i].n_slots;
        L.E = pools[i].E;
        L.layer = layer;
    }
    B.sbytes = slot_bytes(pools[0].H, pools[0].I);
    const int blocks = (hdr.free_sms > 0 ? hdr.free_sms : num_sms()) * 4;
    B.per = blocks / n > 1 ? blocks / n : 1;
    k_cache_plan_batch<<<1, 32, 0, s>>>(B, *c, hdr.pf_plans);
    if (launch_ok() != E0_OK) return E0_ERR_CUDA;
    k_cache_copy_batch<<<n * B.per, 512, 0, s>>>(B, *c, hdr.pf_plans);
    if (launch_ok() != E0_OK) return E0_ERR_CUDA;
    k_slot_commit_batch<<<n, 32, 0, s>>>(B, st);
    return launch_ok();
}

int stack_prefetch_experts_cached(void* ws, int layer, int t_next, const e0_slot_pool* p, const uint8_t* bank,
                                  const e0_expert_cache* c, uint32_t* st, cudaStream_t s) {
    StackHdr hdr;
    if (!stack_hdr(ws, &hdr)) return E0_ERR_ARG;
    if (layer < 0 || layer >= hdr.L || t_next < 1) return E0_ERR_ARG;
    if ((long)(layer + 1) * p->E > c->n_keys) return E0_ERR_ARG;
    const int32_t* next = hdr.pred_inds + ((size_t)(t_next & 1) * hdr.L + layer) * hdr.K;
    k_cache_plan<<<1, 32, 0, s>>>(p->slot_table, p->occupant, p->n_slots, p->E, next, hdr.K, layer, *c);
    k_cache_copy<<<hdr.free_sms > 0 ? hdr.free_sms : num_sms(), 512, 0, s>>>(p->data, bank, *c, slot_bytes(p->H, p->I));
    k_slot_commit<<<1, 32, 0, s>>>(p->slot_table, p->occupant, p->n_slots, p->E, next, hdr.K, nullptr, 0, st);
    return launch_ok();
}

int stack_step(const float* x, float* r_out, void* ws, const e0_stack_trace* trace, int impl, uint32_t* st,
               cudaStream_t s) {
    num_sms();
    StackHdr* Sp = reinterpret_cast<StackHdr*>(ws);
    StackHdr hdr;
    {
        std::lock_guard<std::mutex> g(g_stack_mu);
        auto it = g_stacks.find(ws);
        if (it == g_stacks.end()) return E0_ERR_ARG;
        hdr = it->second;
    }
    TraceP tr;
    memset(&tr, 0, sizeof(tr));
    if (trace) {
        tr.r = trace->r;
        tr.inds = trace->inds;
        tr.w = trace->w;
        tr.head_logits = trace->head_logits;
        tr.pred_inds = trace->pred_inds;
    }
    if (impl == 2) return E0_ERR_UNSUPPORTED;  // retired (the cluster kernel)
    if (impl == 3) return stack_step_ll(x, r_out, ws, hdr, 0, hdr.L, trace, st, s);
    if (impl == 0) {
        const PersistSmem lay(hdr.H, hdr.E, hdr.K, (size_t)hdr.smem);
        void* args[] = {&Sp, (void*)&x, &r_out, &tr, &st};
        return cuda_ok(cudaLaunchCooperativeKernel((const void*)k_stack_token, dim3(hdr.grid), dim3(PHASE_THREADS),
                                                   args, lay.total, s));
    }
    const int H = hdr.H, I = hdr.I, E = hdr.E, K = hdr.K;
    const int R = (H / GROUP) >= 32 ? 1 : 32 / (H / GROUP);
    const size_t gsm = GateUpSmem(1, H, K).total;
    const size_t dsm = DownSmem(1, I, K, true, E0_MAX_LORA_RANK, hdr.hidden > 0 ? hdr.hidden : GROUP).total;
    const int RI = (I / GROUP) >= 32 ? 1 : 32 / (I / GROUP);
    for (int l = 0; l < hdr.L; ++l) {
        k_stack_norm<<<1, 256, 0, s>>>(Sp, l, x, tr);
        k_stack_router<<<phase_grid((long)E / R + 1), PHASE_THREADS, 0, s>>>(Sp, l, st);
        k_stack_resolve<<<1, 32, (size_t)E * 4, s>>>(Sp, l, tr, st);
        k_stack_gateup<<<phase_grid((long)(K + 1) * I / R + 2 * hdr.rank + (hdr.hidden + E) / R), PHASE_THREADS,
                         gsm, s>>>(Sp, l, st);
        k_stack_down<<<phase_grid((long)H / RI + E), PHASE_THREADS, dsm, s>>>(Sp, l, x, r_out, st);
        k_stack_head<<<1, 32, (size_t)E * 4, s>>>(Sp, l, tr, st);
        if (launch_ok() != E0_OK) return E0_ERR_CUDA;
    }
    k_stack_finish<<<1, 256, 0, s>>>(Sp, r_out, tr);
    return launch_ok();
}

}  // namespace e0

// ================================================================== bounded-wait self-test

namespace e0 {

// One thread polls a flag the way every spin of this library does: bounded
// by device time, ending in a status bit instead of a trap.
__global__ void k_bounded_wait(const uint32_t* flag, uint64_t limit_ns, uint32_t* st) {
    if (threadIdx.x != 0) return;
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    while (true) {
        uint32_t v;
        asm volatile("ld.relaxed.gpu.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v) return;
        uint64_t t1;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
        if (t1 - t0 > limit_ns) {
            set_status(st, E0_ST_TIMEOUT);
            return;
        }
        __nanosleep(256);
    }
}

int selftest_bounded_wait(const uint32_t* flag, uint32_t limit_us, uint32_t* st, cudaStream_t s) {
    k_bounded_wait<<<1, 32, 0, s>>>(flag, (uint64_t)limit_us * 1000ull, st);
    return cudaGetLastError() == cudaSuccess ? E0_OK : E0_ERR_CUDA;
}

}  // namespace e0
