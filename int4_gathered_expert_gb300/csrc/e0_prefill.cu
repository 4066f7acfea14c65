// Whole-layer prefill ([PTKR] "SSD 전문가 스트리밍": the full-layer path loads a
// layer's 9 tensors and computes with a sorted gather; [JAEHUN] "작동 원리":
// prefill routes natively and never predicts):
//   1. router logits on the tensor cores (fp16 X, fp16 W_r, fp32 accumulate);
//   2. routing per token; tokens whose top-(K+1) logits are closer than
//      REFINE_GAP get their logits recomputed with fp32 SIMT dot products
//      before routing, so near-ties are decided as accurately as in decode;
//   3. stable counting sort of the T*K assignments by expert;
//   4. gather of the X rows into expert order;
//   5. grouped GEMM gate/up on tcgen05 (int4 weights dequantised on chip into
//      the 128-row M operand, tokens as the N operand), SwiGLU epilogue -> fp16;
//   6. grouped GEMM down, epilogue scales each row by its routing weight and
//      adds it into Y[t] (fp32 atomics: the K terms of a token land in a
//      varying order);
//   7. with E0MOE_PREFILL_FIXED_ORDER=1 the rows go to an fp16 buffer
//      instead and a combine sums a token's K rows in a fixed order.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "e0_decode.cuh"
#include "e0_internal.h"
#include "e0_umma.cuh"

namespace e0 {

constexpr int SEG = 256;            // assignments per sort segment (one block)
constexpr int BM = 128, BK = 64, BN = 128;
constexpr int GEMM_THREADS = 192;   // warps 0-3 dequant + epilogue, 4 TMA, 5 MMA
constexpr int STAGES = 4;
constexpr float REFINE_GAP = 2e-4f;  // well above the error of fp32 tensor-core accumulation over K = H
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s

enum { MODE_GATEUP = 1, MODE_DOWN = 2 };

struct PrefillWs {
    float* logits;      // [T][E]
    int32_t* inds;      // [T][K]
    float* w;           // [T][K]
    int32_t* counts;    // [E]
    int32_t* offsets;   // [E+1]
    int32_t* perm;      // [T*K]  sorted position -> assignment
    int32_t* pos;       // [T*K]  assignment -> sorted position
    int32_t* seg_cnt;   // [nseg][E]
    int32_t* seg_base;  // [nseg][E]
    int4* tiles;        // [max_tiles] {expert, first sorted row, n0, rows}, most rows first
    int32_t* flag;      // [T+1] tokens whose routing is recomputed in fp32 (count first)
    int32_t* done;      // [T] row groups of a flagged token whose exact logits are written
    int32_t* n_tiles;   // [1]
    uint32_t* err;      // [1] timeouts inside the GEMMs
    float* wp;          // [T*K] routing weight per sorted row
    __half* xp;         // [T*K][H] gathered rows
    __half* abuf;       // [T*K][I] SwiGLU activations
    __half* yp;         // [T*K][H] weighted expert outputs (fp16)
    size_t bytes;
    int max_tiles;
};

static PrefillWs prefill_ws(char* base, int T, int H, int I, int E, int K) {
    const size_t A = (size_t)T * K;
    const size_t nseg = (A + SEG - 1) / SEG;
    size_t off = 0;
    auto take = [&](size_t n) {
        off = (off + 255) & ~(size_t)255;
        char* p = base + off;
        off += n;
        return p;
    };
    PrefillWs w;
    w.max_tiles = (int)((A + BN - 1) / BN) + E;
    w.logits = reinterpret_cast<float*>(take((size_t)T * E * 4));
    w.inds = reinterpret_cast<int32_t*>(take(A * 4));
    w.w = reinterpret_cast<float*>(take(A * 4));
    w.counts = reinterpret_cast<int32_t*>(take((size_t)E * 4));
    w.offsets = reinterpret_cast<int32_t*>(take((size_t)(E + 1) * 4));
    w.perm = reinterpret_cast<int32_t*>(take(A * 4));
    w.pos = reinterpret_cast<int32_t*>(take(A * 4));
    w.seg_cnt = reinterpret_cast<int32_t*>(take(nseg * E * 4));
    w.seg_base = reinterpret_cast<int32_t*>(take(nseg * E * 4));
    w.tiles = reinterpret_cast<int4*>(take((size_t)w.max_tiles * 16));
    w.flag = reinterpret_cast<int32_t*>(take((size_t)(T + 1) * 4));
    w.done = reinterpret_cast<int32_t*>(take((size_t)T * 4));
    w.n_tiles = reinterpret_cast<int32_t*>(take(16));
    w.err = reinterpret_cast<uint32_t*>(take(16));
    w.wp = reinterpret_cast<float*>(take(A * 4));
    w.xp = reinterpret_cast<__half*>(take(A * H * 2));
    w.abuf = reinterpret_cast<__half*>(take(A * I * 2));
    w.yp = reinterpret_cast<__half*>(take(A * H * 2));
    w.bytes = off + 256;
    return w;
}

size_t prefill_ws_bytes(int T, int H, int I, int E, int K) { return prefill_ws(nullptr, T, H, I, E, K).bytes; }

// ------------------------------------------------------------------ stable counting sort

__global__ void k_sort_hist(const int32_t* inds, int A, int E, int32_t* seg_cnt) {
    extern __shared__ int32_t cnt[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int a = blockIdx.x * SEG + threadIdx.x;
    if (a < A) {
        const int e = inds[a];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) seg_cnt[(size_t)blockIdx.x * E + e] = cnt[e];
}

// one block of 1024 threads: totals, exclusive scan over experts, per-segment
// bases.  Q = blockDim / E threads share an expert: thread (q, e) walks the
// segments [q nseg / Q, (q + 1) nseg / Q), so an expert's global loads run
// Q at a time instead of one after another.
__global__ void k_sort_scan(const int32_t* seg_cnt, int nseg, int E, int32_t* counts, int32_t* offsets,
                            int32_t* seg_base) {
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t part[1024];   // [q][e] count of expert e over thread (q, e)'s segments
    __shared__ int32_t base_e[1024]; // exclusive scan of the totals
    const int Q = max(1, (int)blockDim.x / E);
    const int x = threadIdx.x, pe = x % E, q = x / E;
    const bool walker = x < Q * E;
    const int s0 = q * nseg / Q, s1 = (q + 1) * nseg / Q;
    int pc = 0;
    if (walker)
        for (int s = s0; s < s1; ++s) pc += seg_cnt[(size_t)s * E + pe];
    part[x] = pc;
    __syncthreads();
    const int e = threadIdx.x;
    int c = 0;
    if (e < E)
        for (int j = 0; j < Q; ++j) c += part[j * E + e];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        warp_tot[lane] = v;
    }
    __syncthreads();
    const int excl = incl - c + (warp > 0 ? warp_tot[warp - 1] : 0);
    if (e < E) {
        counts[e] = c;
        offsets[e] = excl;
        base_e[e] = excl;
    }
    if (e == E - 1) offsets[E] = excl + c;
    __syncthreads();
    if (walker) {
        int base = base_e[pe];
        for (int j = 0; j < q; ++j) base += part[j * E + pe];
        for (int s = s0; s < s1; ++s) {
            seg_base[(size_t)s * E + pe] = base;
            base += seg_cnt[(size_t)s * E + pe];
        }
    }
}

__global__ void k_sort_scatter(const int32_t* inds, int A, int E, const int32_t* seg_base, int32_t* perm,
                               int32_t* pos) {
    __shared__ int32_t ex[SEG];
    const int a = blockIdx.x * SEG + threadIdx.x;
    const int e = a < A ? inds[a] : -1;
    ex[threadIdx.x] = e;
    __syncthreads();
    if (a >= A || e < 0 || e >= E) return;
    int rank = 0;
    for (int j = 0; j < (int)threadIdx.x; ++j) rank += ex[j] == e;
    const int p = seg_base[(size_t)blockIdx.x * E + e] + rank;
    perm[p] = a;
    if (pos) pos[a] = p;
}

static int sort_into(const int32_t* inds, int T, int K, int E, int32_t* counts, int32_t* offsets, int32_t* perm,
                     int32_t* pos, const PrefillWs& w, cudaStream_t s) {
    const int A = T * K;
    const int nseg = (A + SEG - 1) / SEG;
    if (A == 0) {
        if (cudaMemsetAsync(counts, 0, (size_t)E * 4, s) != cudaSuccess) return E0_ERR_CUDA;
        if (cudaMemsetAsync(offsets, 0, (size_t)(E + 1) * 4, s) != cudaSuccess) return E0_ERR_CUDA;
        return E0_OK;
    }
    k_sort_hist<<<nseg, SEG, (size_t)E * 4, s>>>(inds, A, E, w.seg_cnt);
    k_sort_scan<<<1, 1024, 0, s>>>(w.seg_cnt, nseg, E, counts, offsets, w.seg_base);
    k_sort_scatter<<<nseg, SEG, 0, s>>>(inds, A, E, w.seg_base, perm, pos);
    return cudaGetLastError() == cudaSuccess ? E0_OK : E0_ERR_CUDA;
}

int prefill_sort(const int32_t* inds, int T, int K, int E, int32_t* counts, int32_t* offsets, int32_t* perm,
                 void* ws, cudaStream_t s) {
    const PrefillWs w = prefill_ws(reinterpret_cast<char*>(ws), T, 64, 64, E, K);
    return sort_into(inds, T, K, E, counts, offsets, perm, nullptr, w, s);
}

// ------------------------------------------------------------------ tcgen05 GEMM

struct GemmP {
    int K;              // reduction length (elements)
    int rows_out;       // rows of A that exist (E for the router, I for gate/up, H for down)
    // router
    int T;
    float* logits;
    int E;
    // grouped
    const uint8_t* pool;
    const int32_t* table;
    int n_slots;
    size_t slot_bytes;
    int H, I;
    const int4* tiles;
    const int32_t* n_tiles;
    __half* abuf;
    __half* yp;
    const float* wp;
    const int32_t* perm;   // sorted row -> assignment t*K + k
    float* Y;              // [T][H]: the down epilogue adds into it (accumulate != 0)
    int Kr;                // experts per token
    int accumulate;        // 1: atomic adds into Y; 0: fp16 rows into yp, then the combine
    uint32_t* err;
    uint32_t* st;
};

// Router GEMM: logits[T][E] = X W_r^T on the tensor cores.  One CTA computes
// one 128-row (experts) x BN-column (tokens) output tile.  Roles:
//   warps 0-3  drain the accumulator from TMEM (thread t owns TMEM lane t);
//   warp 4     issues the TMA loads of both operand tiles;
//   warp 5     allocates TMEM and, from one thread, issues tcgen05.mma.
// Pipeline: STAGES shared-memory stages guarded by full/empty mbarriers; the
// MMA thread frees a stage with tcgen05.commit.  Every wait is time-bounded:
// on timeout the CTA raises *err, stops its loops, frees TMEM and returns.
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    k_router_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmP p) {
    constexpr uint32_t A_BYTES = BM * BK * 2;
    constexpr uint32_t B_BYTES = BN * BK * 2;
    constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    constexpr uint32_t TMEM_COLS = BN;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BM;
    const int row0 = blockIdx.y * BN;
    const int ncount = min(BN, p.T - row0);
    if (ncount <= 0) return;
    const int n_mma = (ncount + 15) & ~15;
    const int nk = p.K / BK;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* accum = empty + STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
    volatile uint32_t* abort = tmem_slot + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accum, 1);
        *abort = 0;
        mbar_fence_init();
    }
    if (warp == 5) tmem_alloc(tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        // ---------------- epilogue: TMEM -> registers -> global
        const bool have = mbar_wait(accum, 0, abort, WAIT_LIMIT_NS);
        if (!have) {
            *abort = 1;
            atomicOr(p.err, 2u);
        }
        tc_fence_after();
        const int r = warp * 32 + lane;
        const int row = m0 + r;
        const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16);
        for (int c0 = 0; c0 < n_mma && have; c0 += 16) {
            float acc[16];
            tmem_ld16(tbase + c0, acc);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int col = c0 + j;
                if (col < ncount && row < p.rows_out) p.logits[(size_t)(row0 + col) * p.E + row] = acc[j];
            }
        }
    } else if (warp == 4) {
        // ---------------- TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmB);
            tma_prefetch_desc(&tmA);
            for (int kk = 0; kk < nk; ++kk) {
                const int s = kk % STAGES;
                if (!mbar_wait(&empty[s], ((kk / STAGES) + 1) & 1, abort, WAIT_LIMIT_NS)) {
                    *abort = 1;
                    atomicOr(p.err, 4u);
                    break;
                }
                uint8_t* st = smem + s * STAGE_BYTES;
                mbar_arrive_expect_tx(&full[s], B_BYTES + A_BYTES);
                tma_load_2d(&tmB, &full[s], st + A_BYTES, kk * BK, row0);
                tma_load_2d(&tmA, &full[s], st, kk * BK, m0);
            }
        }
    } else {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(BM, n_mma);
            bool ok = true;
            for (int kk = 0; kk < nk; ++kk) {
                const int s = kk % STAGES;
                if (!mbar_wait(&full[s], (kk / STAGES) & 1, abort, WAIT_LIMIT_NS)) {
                    *abort = 1;
                    atomicOr(p.err, 8u);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = smem_u32(smem + s * STAGE_BYTES);
                const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                for (int j = 0; j < BK / 16; ++j)
                    umma_f16(tmem, sdesc_k_sw128(a_addr + j * 32), sdesc_k_sw128(b_addr + j * 32), idesc, (kk | j) != 0);
                umma_commit(&empty[s]);
            }
            if (ok) umma_commit(accum);
        }
    }
    // drain: make sure no TMA write or MMA read of this CTA's shared memory is
    // still in flight before the CTA exits (bounded by the same limit)
    if (threadIdx.x == 160 && *abort) {
        for (int s = 0; s < STAGES; ++s) mbar_wait(&empty[s], 0, abort, 1000000ull);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

static size_t router_gemm_smem() { return (size_t)STAGES * (BM * BK * 2 + BN * BK * 2) + 1024 + 256; }

// ------------------------------------------------------------------ persistent grouped GEMM with TMA-fed dequant

// One CTA per SM loops over work items (tile of up to P2_BN tokens of one
// expert x one 128-row slice of its weights).  Per K step the weight tile
// goes HBM -> shared memory (raw int4 codes, 4 KB) -> registers -> tensor
// memory (fp16, the MMA's A operand), so the dequantised tile costs no
// shared-memory bandwidth; the token tile (B operand) is a TMA load into
// shared memory.  Rings: raw code tiles P2_RAW_STAGES deep, operand stages
// (A columns in tensor memory, B tile in shared memory) P2_OP_STAGES deep.
// Roles:
//   warps 0-3, 11-14  dequantise (two groups taking alternate K steps): thread
//              r turns row r of a raw tile into fp16 and stores it into
//              tensor-memory lane r of an operand stage;
//   warps 4-7  epilogue: drain one of two TMEM accumulators while the MMA
//              fills the other;
//   warp 8     TMA: raw code tiles (tensor map over the slot pool), running
//              up to P2_RAW_STAGES K steps ahead;
//   warp 9     TMEM allocation and the tcgen05.mma issue;
//   warp 10    TMA: token tiles into the operand stages.
// In the gate/up GEMM a 128-row slice is 64 intermediate rows with the gate
// and up rows interleaved (the slot layout stores them that way), so each
// SwiGLU pair sits in adjacent TMEM lanes.
constexpr int P2_BK = 128;           // K of one pipeline step (eight MMAs of K = 16)
constexpr int P2_OP_STAGES = 4;
constexpr int P2_RAW_STAGES = 8;
constexpr int P2_THREADS = 480;
constexpr int P2_BN = 128;
constexpr uint32_t P2_B = P2_BN * 128;     // token tile of 64 k (one 128B-swizzled TMA box)
constexpr uint32_t P2_RAW = 128 * P2_BK / 2;  // raw int4 codes of one K step
constexpr uint32_t P2_OP = 2 * P2_B;       // shared memory of an operand stage: two token tiles
constexpr uint32_t P2_ACOL = 2 * P2_BN;    // first tensor-memory column of the A tiles (after two accumulators)

struct P2Item {
    int slot, row0, ncount, m;
};

// The item a CTA takes in round k: round-robin over the CTAs, in alternating
// directions, so that the heaviest items (first in the tile order) spread
// evenly.  Later rounds hold larger positions, so a CTA stops at the first
// position past the last item.
E0_DEV int p2_pos(int k) {
    const int G = gridDim.x, c = blockIdx.x;
    return k * G + ((k & 1) ? G - 1 - c : c);
}

E0_DEV P2Item p2_item(const GemmP& p, int idx, int MT) {
    const int4 tl = p.tiles[idx / MT];
    P2Item it;
    it.m = idx % MT;
    it.row0 = tl.y;
    it.ncount = tl.w;
    const int s = (tl.x >= 0 && tl.x < p.E) ? p.table[tl.x] : -1;
    it.slot = (s >= 0 && s < p.n_slots) ? s : -1;
    return it;
}

E0_DEV void tma_load_4d(const CUtensorMap* map, uint64_t* bar, void* dst, int x, int y, int z, int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
        : "memory");
}

E0_DEV void tma_load_5d(const CUtensorMap* map, uint64_t* bar, void* dst, int x, int y, int z, int w, int v) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5, %6}], [%7];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(v), "r"(smem_u32(bar))
        : "memory");
}

E0_DEV void tma_load_3d(const CUtensorMap* map, uint64_t* bar, void* dst, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// SiLU for the gate/up epilogue, from CUDA's fast exponential and division
// intrinsics (relative error ~1e-7, far below the fp16 rounding of the
// result): x * sigmoid(x) = x / (1 + e^-x); for x -> -inf the divisor
// overflows and the quotient goes to 0, for x -> +inf it is x.
E0_DEV float silu_fast(float x) { return __fdividef(x, 1.f + __expf(-x)); }

template <int MODE>
__global__ void __launch_bounds__(P2_THREADS, 1)
    k_umma2(const __grid_constant__ CUtensorMap tmCodes, const __grid_constant__ CUtensorMap tmB, GemmP p) {
    // two fp32 accumulators of P2_BN columns, then one 32-column fp16 A tile
    // (128 rows x 64 k) per operand stage
    constexpr uint32_t TMEM_COLS = 512;
    static_assert(P2_ACOL + (P2_BK / 2) * P2_OP_STAGES <= TMEM_COLS, "tensor-memory columns");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int MT = MODE == MODE_GATEUP ? (2 * p.I) / 128 : p.H / 128;
    const int n_items = *p.n_tiles * MT;
    const int nk = p.K / P2_BK;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* raw_ring = smem + P2_OP_STAGES * P2_OP;
    uint64_t* raw_full = reinterpret_cast<uint64_t*>(raw_ring + P2_RAW_STAGES * P2_RAW);
    uint64_t* raw_empty = raw_full + P2_RAW_STAGES;
    uint64_t* a_full = raw_empty + P2_RAW_STAGES;
    uint64_t* b_full = a_full + P2_OP_STAGES;
    uint64_t* op_empty = b_full + P2_OP_STAGES;
    uint64_t* acc_full = op_empty + P2_OP_STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    volatile uint32_t* abort = tmem_slot + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P2_RAW_STAGES; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], 4);  // one arrival per dequantising warp
        }
        for (int s = 0; s < P2_OP_STAGES; ++s) {
            mbar_init(&a_full[s], 4);
            mbar_init(&b_full[s], 1);
            mbar_init(&op_empty[s], 1);
        }
        for (int b2 = 0; b2 < 2; ++b2) {
            mbar_init(&acc_full[b2], 1);
            mbar_init(&acc_empty[b2], 128);
        }
        *abort = 0;
        mbar_fence_init();
    }
    if (warp == 9) tmem_alloc(tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const SlotLayout sl{p.H, p.I};
    // a producer that stops early waits (bounded, abort flag ignored) for the
    // copies it issued before the block can leave
    const volatile uint32_t never = 0;

    if (warp < 4 || warp >= 11) {
        // ---------------- dequantisers: two groups of four warps take alternate
        // K steps (warps 0-3 the even global steps, 11-14 the odd ones), so that
        // one step's load -> convert -> tensor-memory store chain overlaps the
        // other's; thread r handles weight row r, tensor-memory lane r
        const int grp = warp < 4 ? 0 : 1;
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;
        uint32_t gbase = 0;  // global step of the item's first K step
        bool ok = true;
        for (int k = 0, idx; (idx = p2_pos(k)) < n_items && ok; ++k) {
            const P2Item it = p2_item(p, idx, MT);
            const uint8_t* ex = it.slot >= 0 ? p.pool + (size_t)it.slot * p.slot_bytes : nullptr;
            const int wr = it.m * 128 + r;  // weight row (interleaved gate/up rows for MODE_GATEUP)
            const uint8_t* sbp = nullptr;
            if (ex) {
                if (MODE == MODE_GATEUP) sbp = ex + sl.gu_sb() + (size_t)wr * (p.H / GROUP) * 4;
                else sbp = ex + sl.down_sb_off(wr, 0);  // group kk at + kk * DROWS * 4
            }
            const size_t sstep = MODE == MODE_GATEUP ? (size_t)4 : (size_t)DROWS * 4;
            // this group's steps of the item: kk = kk0, kk0 + 2, ...
            const int kk0 = (int)((gbase + (uint32_t)grp) & 1u);
            const int n_own = nk > kk0 ? (nk - kk0 + 1) / 2 : 0;
            // (scale, bias) words of 4 own steps (two 64-groups each) are loaded
            // one chunk ahead of use
            uint32_t sbw[4][2], sbn[4][2];
#pragma unroll
            for (int d = 0; d < 4; ++d)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    sbn[d][h] = (ex && d < n_own) ? ldg_u32(sbp + (size_t)(2 * (kk0 + 2 * d) + h) * sstep) : 0u;
            for (int i0 = 0; i0 < n_own && ok; i0 += 4) {
#pragma unroll
                for (int d = 0; d < 4; ++d) {
                    const int in = i0 + 4 + d;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        sbw[d][h] = sbn[d][h];
                        sbn[d][h] = (ex && in < n_own) ? ldg_u32(sbp + (size_t)(2 * (kk0 + 2 * in) + h) * sstep) : 0u;
                    }
                }
#pragma unroll
                for (int d = 0; d < 4; ++d) {
                    const int i = i0 + d;
                    if (i >= n_own) break;
                    const uint32_t g = gbase + (uint32_t)(kk0 + 2 * i);
                    const uint32_t rs = g % P2_RAW_STAGES, os = g % P2_OP_STAGES;
                    const bool w = mbar_wait(&raw_full[rs], (g / P2_RAW_STAGES) & 1, abort, WAIT_LIMIT_NS) &&
                                   mbar_wait(&op_empty[os], ((g / P2_OP_STAGES) + 1) & 1, abort, WAIT_LIMIT_NS);
                    if (!__all_sync(0xffffffffu, w)) {  // the warp leaves together
                        ok = false;
                        *abort = 1;
                        atomicOr(p.err, 16u);
                        break;
                    }
                    tc_fence_after();
                    // gate/up raw tile: [128 rows][64 B]; down raw tile: [8 row
                    // blocks][4 half-groups][16 rows][16 B]
                    const uint8_t* raw = raw_ring + rs * P2_RAW;
                    const uint8_t* rd = raw + ((r / DROWS) * 4 * DROWS + r % DROWS) * 16;
                    const uint32_t acol = tmem + ((uint32_t)(q4 * 32) << 16) + P2_ACOL + os * (P2_BK / 2);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {  // the two 64-input groups of the step
                        uint32_t o[32];
                        if (ex) {
                            const uint4 c0 = *reinterpret_cast<const uint4*>(
                                MODE == MODE_GATEUP ? raw + r * 64 + h * 32 : rd + 2 * h * DROWS * 16);
                            const uint4 c1 = *reinterpret_cast<const uint4*>(
                                MODE == MODE_GATEUP ? raw + r * 64 + h * 32 + 16 : rd + (2 * h + 1) * DROWS * 16);
                            dequant64_to_regs(c0, c1, sbw[d][h], o);
                        } else {
#pragma unroll
                            for (int c = 0; c < 32; ++c) o[c] = 0u;
                        }
                        tmem_st32(acol + h * 32, o);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    // once every lane is here, the warp has also used the values it
                    // read from the raw slot (an arrive does not order those
                    // generic-proxy reads before the next TMA write into the slot)
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&raw_empty[rs]);
                        mbar_arrive(&a_full[os]);
                    }
                }
            }
            gbase += (uint32_t)nk;
        }
    } else if (warp < 8) {
        // ---------------- epilogue
        const int q = threadIdx.x - 128;  // TMEM lane
        const uint32_t tq = tmem + ((uint32_t)((warp - 4) * 32) << 16);
        uint32_t ii = 0;
        for (int k = 0, idx; (idx = p2_pos(k)) < n_items; ++k, ++ii) {
            const P2Item it = p2_item(p, idx, MT);
            const uint32_t buf = ii & 1;
            const bool have = mbar_wait(&acc_full[buf], (ii >> 1) & 1, abort, WAIT_LIMIT_NS);
            if (!have) {
                *abort = 1;
                atomicOr(p.err, 32u);
            }
            tc_fence_after();
            const int n_mma = (it.ncount + 15) & ~15;
            // per item: the output base of this lane's row; per 32 columns: two
            // tensor-memory loads, one wait
            __half* hout = nullptr;
            __half* yout = nullptr;
            if (MODE == MODE_GATEUP) hout = p.abuf + (size_t)it.row0 * p.I + it.m * 64 + (q >> 1);
            else yout = p.yp + (size_t)it.row0 * p.H + it.m * 128 + q;
            float* yacc = p.Y + it.m * 128 + q;  // accumulate: row t of Y at + t * H
            for (int c0 = 0; c0 < n_mma && have; c0 += 32) {
                float acc[32];
                tmem_ld16(tq + buf * P2_BN + c0, *reinterpret_cast<float(*)[16]>(acc));
                const bool two = c0 + 16 < n_mma;  // warp-uniform
                if (two) tmem_ld16(tq + buf * P2_BN + c0 + 16, *reinterpret_cast<float(*)[16]>(acc + 16));
                else
#pragma unroll
                    for (int j = 16; j < 32; ++j) acc[j] = 0.f;
                tmem_ld_wait();
                if (MODE == MODE_GATEUP) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float other = __shfl_xor_sync(0xffffffffu, acc[j], 1);
                        const int col = c0 + j;
                        if (!(q & 1) && col < it.ncount)
                            hout[(size_t)col * p.I] = __float2half_rn(silu_fast(acc[j]) * other);
                    }
                } else {
                    // the routing weights (and, accumulating, the tokens) of these
                    // 32 columns, one per lane
                    const bool lv = c0 + lane < it.ncount;
                    const float wl = lv ? p.wp[it.row0 + c0 + lane] : 0.f;
                    if (p.accumulate) {
                        const int tl = lv ? p.perm[it.row0 + c0 + lane] / p.Kr : 0;
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int col = c0 + j;
                            const float wj = __shfl_sync(0xffffffffu, wl, j);
                            const int tj = __shfl_sync(0xffffffffu, tl, j);
                            if (col < it.ncount) atomicAdd(yacc + (size_t)tj * p.H, wj * acc[j]);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int col = c0 + j;
                            const float wj = __shfl_sync(0xffffffffu, wl, j);
                            if (col < it.ncount) yout[(size_t)col * p.H] = __float2half_rn(wj * acc[j]);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[buf]);
            if (!have) break;
        }
    } else if (warp == 8) {
        // ---------------- TMA: raw code tiles, up to P2_RAW_STAGES steps ahead
        if (lane == 0) {
            tma_prefetch_desc(&tmCodes);
            uint32_t g = 0;
            bool ok = true;
            for (int k = 0, idx; (idx = p2_pos(k)) < n_items && ok; ++k) {
                const P2Item it = p2_item(p, idx, MT);
                const int z = it.slot >= 0 ? it.slot : 0;
                for (int kk = 0; kk < nk; ++kk, ++g) {
                    const uint32_t rs = g % P2_RAW_STAGES;
                    if (!mbar_wait(&raw_empty[rs], ((g / P2_RAW_STAGES) + 1) & 1, abort, WAIT_LIMIT_NS)) {
                        ok = false;
                        *abort = 1;
                        atomicOr(p.err, 64u);
                        break;
                    }
                    uint8_t* dst = raw_ring + rs * P2_RAW;
                    mbar_arrive_expect_tx(&raw_full[rs], P2_RAW);
                    if (MODE == MODE_GATEUP) tma_load_3d(&tmCodes, &raw_full[rs], dst, kk * (P2_BK / 2), it.m * 128, z);
                    else tma_load_5d(&tmCodes, &raw_full[rs], dst, 0, 0, 4 * kk, it.m * (128 / DROWS), z);
                }
            }
            // the copies issued into each slot have landed before the block leaves
            for (uint32_t d = 0; d < P2_RAW_STAGES && d < g; ++d) {
                const uint32_t gl = g - 1 - d;
                mbar_wait(&raw_full[gl % P2_RAW_STAGES], (gl / P2_RAW_STAGES) & 1, &never, WAIT_LIMIT_NS);
            }
        }
    } else if (warp == 10) {
        // ---------------- TMA: token tiles into the operand stages
        if (lane == 0) {
            tma_prefetch_desc(&tmB);
            uint32_t g = 0;
            bool ok = true;
            for (int k = 0, idx; (idx = p2_pos(k)) < n_items && ok; ++k) {
                const P2Item it = p2_item(p, idx, MT);
                for (int kk = 0; kk < nk; ++kk, ++g) {
                    const uint32_t os = g % P2_OP_STAGES;
                    if (!mbar_wait(&op_empty[os], ((g / P2_OP_STAGES) + 1) & 1, abort, WAIT_LIMIT_NS)) {
                        ok = false;
                        *abort = 1;
                        atomicOr(p.err, 512u);
                        break;
                    }
                    mbar_arrive_expect_tx(&b_full[os], 2 * P2_B);
                    tma_load_2d(&tmB, &b_full[os], smem + os * P2_OP, kk * P2_BK, it.row0);
                    tma_load_2d(&tmB, &b_full[os], smem + os * P2_OP + P2_B, kk * P2_BK + 64, it.row0);
                }
            }
            for (uint32_t d = 0; d < P2_OP_STAGES && d < g; ++d) {
                const uint32_t gl = g - 1 - d;
                mbar_wait(&b_full[gl % P2_OP_STAGES], (gl / P2_OP_STAGES) & 1, &never, WAIT_LIMIT_NS);
            }
        }
    } else {
        // ---------------- MMA issuer
        if (lane == 0) {
            uint32_t g = 0, ii = 0;
            bool ok = true;
            for (int k = 0, idx; (idx = p2_pos(k)) < n_items && ok; ++k, ++ii) {
                const P2Item it = p2_item(p, idx, MT);
                const uint32_t buf = ii & 1;
                if (!mbar_wait(&acc_empty[buf], ((ii >> 1) + 1) & 1, abort, WAIT_LIMIT_NS)) {
                    *abort = 1;
                    atomicOr(p.err, 128u);
                    break;
                }
                tc_fence_after();
                const int n_mma = (it.ncount + 15) & ~15;
                const uint32_t idesc = idesc_f16_f32(128, n_mma);
                for (int kk = 0; kk < nk; ++kk, ++g) {
                    const uint32_t os = g % P2_OP_STAGES;
                    const uint32_t ph = (g / P2_OP_STAGES) & 1;
                    if (!mbar_wait(&b_full[os], ph, abort, WAIT_LIMIT_NS) ||
                        !mbar_wait(&a_full[os], ph, abort, WAIT_LIMIT_NS)) {
                        ok = false;
                        *abort = 1;
                        atomicOr(p.err, 256u);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t b_addr = smem_u32(smem + os * P2_OP);
                    const uint32_t a_tm = tmem + P2_ACOL + os * (P2_BK / 2);
#pragma unroll
                    for (int j = 0; j < P2_BK / 16; ++j)
                        umma_f16_ta(tmem + buf * P2_BN, a_tm + j * 8,
                                    sdesc_k_sw128(b_addr + (j >> 2) * P2_B + (j & 3) * 32), idesc, (kk | j) != 0);
                    umma_commit(&op_empty[os]);
                }
                if (!ok) break;
                umma_commit(&acc_full[buf]);
            }
            // the MMAs issued have completed before TMEM is freed
            if (g > 0) {
                const uint32_t gl = g - 1;
                mbar_wait(&op_empty[gl % P2_OP_STAGES], (gl / P2_OP_STAGES) & 1, &never, WAIT_LIMIT_NS);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

static size_t gemm2_smem() {
    return (size_t)P2_OP_STAGES * P2_OP + (size_t)P2_RAW_STAGES * P2_RAW +
           (2 * P2_RAW_STAGES + 3 * P2_OP_STAGES + 4) * 8 + 8 + 1024;
}

// ------------------------------------------------------------------ small prefill kernels

// Route one token per warp from the tensor-core logits and flag the tokens
// whose routing a logit error below REFINE_GAP could change: the selection
// runs one round past K (and, in group-limited routing, one past G groups)
// and a token is flagged where two consecutive scores of the K + 1 largest,
// or the G-th and (G+1)-th group scores, are closer than that.  A group score
// (the sum of a group's two largest sigmoids) moves by at most half the logit
// error (sigmoid' <= 1/4, two terms), so one threshold serves both gaps.
// MAXM = ceil(E / 32) keys a lane.
template <int MAXM>
__global__ void __launch_bounds__(256) k_prefill_route(const float* logits, int T, int E, RouteP rp, int32_t* inds,
                                                       float* w, int32_t* flag, int32_t* done, uint32_t* st) {
    extern __shared__ float scr[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x * (blockDim.x >> 5) + warp;
    if (t >= T) return;
    const float gap = route_warp_t<MAXM, true>(logits + (size_t)t * E, E, rp, inds + (size_t)t * rp.K,
                                               w + (size_t)t * rp.K, scr + warp * E, st, lane);
    // a group count the ranking does not expect is always refined
    const bool odd = rp.mode == E0_ROUTE_SIGMOID_GROUP && (rp.n_groups < 1 || rp.n_groups > 32 || E % rp.n_groups);
    if (lane == 0 && (odd || !(gap >= REFINE_GAP))) {
        const int i = atomicAdd(flag, 1);
        flag[1 + i] = t;
        done[i] = 0;
    }
}

// fp16 row slice (64 halves) . fp16 x slice (64 halves), fp32 accumulation
E0_DEV float hh64_dot(const __half* wrow, const __half* x) {
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 wv = ldg_stream(wrow + 8 * c);
        const uint4 xv = *reinterpret_cast<const uint4*>(x + 8 * c);
        const __half2* xh = reinterpret_cast<const __half2*>(&xv);
        float xs[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(xh[i]);
            xs[2 * i] = f.x;
            xs[2 * i + 1] = f.y;
        }
        acc += h8_dot(wv, xs);
    }
    return acc;
}

// Exact (fp32 SIMT) logits of the flagged tokens, one warp per (token, row
// group).  Each warp counts the row group it has written into done[i]; the
// warp that completes token i's last one routes the token again from the
// completed row (stores, fence, warp barrier, count: the fenced stores of
// every lane come before the count another warp sees).  Four blocks an SM:
// the grid is four blocks per SM.
template <int MAXM>
__global__ void __launch_bounds__(256, 4) k_prefill_refine(const __half* X, int H, const __half* W_r, int E, RouteP rp,
                                                        const int32_t* flag, int32_t* done, float* logits,
                                                        int32_t* inds, float* w, uint32_t* st) {
    extern __shared__ float scr[];
    const int n = flag[0];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const RowMap rm(H, lane);
    const int per_tok = (E + rm.R - 1) / rm.R;
    const long total = (long)n * per_tok;
    for (long task = (long)blockIdx.x * 8 + warp; task < total; task += (long)gridDim.x * 8) {
        const int i = (int)(task / per_tok);
        const int t = flag[1 + i];
        const int e = (int)(task % per_tok) * rm.R + rm.r;
        float acc = 0.f;
        if (rm.active && e < E) acc = hh64_dot(W_r + (size_t)e * H + GROUP * rm.g, X + (size_t)t * H + GROUP * rm.g);
        acc = seg_sum(acc, rm.G, lane);
        if (rm.active && rm.g == 0 && e < E) logits[(size_t)t * E + e] = acc;
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(&done[i], 1) == per_tok - 1;
        if (__shfl_sync(0xffffffffu, last, 0)) {
            __threadfence();
            route_warp_t<MAXM>(logits + (size_t)t * E, E, rp, inds + (size_t)t * rp.K, w + (size_t)t * rp.K,
                               scr + warp * E, st, lane);
            __syncwarp();
        }
    }
}

// Both routing kernels, instantiated for the keys a lane holds (E / 32
// rounded up to a power of two), so that no instance carries the registers
// of a larger E.
static void launch_route(bool refine, const float* logits_in, float* logits, const __half* X, int H,
                         const __half* W_r, int T, int E, const RouteP& rp, int32_t* flag, int32_t* done,
                         int32_t* inds, float* w, uint32_t* st, cudaStream_t s) {
    const size_t sm = (size_t)8 * E * 4;
#define E0_ROUTE_LAUNCH(M)                                                                                      \
    do {                                                                                                        \
        if (refine)                                                                                             \
            k_prefill_refine<M><<<num_sms() * 4, 256, sm, s>>>(X, H, W_r, E, rp, flag, done, logits, inds, w,  \
                                                               st);                                             \
        else                                                                                                    \
            k_prefill_route<M><<<(T + 7) / 8, 256, sm, s>>>(logits_in, T, E, rp, inds, w, flag, done, st);      \
    } while (0)
    if (E <= 32) E0_ROUTE_LAUNCH(1);
    else if (E <= 64) E0_ROUTE_LAUNCH(2);
    else if (E <= 128) E0_ROUTE_LAUNCH(4);
    else if (E <= 256) E0_ROUTE_LAUNCH(8);
    else if (E <= 512) E0_ROUTE_LAUNCH(16);
    else E0_ROUTE_LAUNCH(32);
#undef E0_ROUTE_LAUNCH
}

// tiles of up to BN consecutive sorted rows of one expert: {e, first row, n0, rows}
__global__ void k_prefill_tiles(const int32_t* counts, const int32_t* offsets, int E, int4* tiles,
                                int32_t* n_tiles) {
    // tiles of up to BN consecutive sorted rows of one expert, heaviest
    // first: every full tile (BN rows) in expert order, then each expert's
    // partial tile by rows, most first (ties to the lower expert).  The
    // grouped GEMMs hand their items out in this order, in alternating
    // directions, so that the CTAs get similar loads.
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t part_rows[1024];
    __shared__ int32_t part_rank[1024];
    const int e = threadIdx.x;
    const int c = e < E ? counts[e] : 0;
    const int nfull = c / BN, rem = c % BN;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    part_rows[e] = rem;
    part_rank[e] = 0;
    // exclusive scan of the full tiles over the experts
    int incl = nfull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        warp_tot[lane] = v;
    }
    __syncthreads();
    const int start = incl - nfull + (warp > 0 ? warp_tot[warp - 1] : 0);
    const int n_full = warp_tot[(blockDim.x - 1) >> 5];
    for (int j = 0; j < nfull; ++j) tiles[start + j] = make_int4(e, offsets[e] + j * BN, j * BN, BN);
    // rank of each partial tile: the partial tiles with more rows, and those
    // with as many of a lower expert, come first.  Q = blockDim / E threads
    // share an expert's count, each over E / Q of the others.
    const int Q = max(1, (int)blockDim.x / E);
    if ((int)threadIdx.x < Q * E) {
        const int pe = threadIdx.x % E, q = threadIdx.x / E;
        const int rem_e = part_rows[pe];
        if (rem_e > 0) {
            int r = 0;
            for (int f = q * E / Q; f < (q + 1) * E / Q; ++f) {
                const int rf = part_rows[f];
                r += rf > rem_e || (rf == rem_e && f < pe);
            }
            if (r) atomicAdd(&part_rank[pe], r);
        }
    }
    const int n_part = __syncthreads_count(rem > 0);
    if (rem > 0) tiles[n_full + part_rank[e]] = make_int4(e, offsets[e] + nfull * BN, nfull * BN, rem);
    if (threadIdx.x == 0) *n_tiles = n_full + n_part;
}

// xp[p] = X[token of perm[p]], wp[p] = w[perm[p]]
__global__ void k_prefill_gather(const __half* X, int H, int K, const int32_t* perm, const float* w, int A,
                                 __half* xp, float* wp) {
    const int row = blockIdx.x;
    if (row >= A) return;
    const int a = perm[row];
    const int t = a / K;
    if (threadIdx.x == 0) wp[row] = w[a];
    const uint4* src = reinterpret_cast<const uint4*>(X + (size_t)t * H);
    uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)row * H);
    for (int c = threadIdx.x; c < H / 8; c += blockDim.x) dst[c] = src[c];
}

// Y[t] = sum_k yp[pos[t*K + k]]  (k = 0..K-1, fixed order, fp32 sums of the
// fp16 rows)
__global__ void k_prefill_combine(const __half* yp, const int32_t* pos, int T, int K, int H, float* Y) {
    const int t = blockIdx.x;
    for (int j = threadIdx.x * 4; j < H; j += blockDim.x * 4) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < K; ++k) {
            const uint2 v = *reinterpret_cast<const uint2*>(yp + (size_t)pos[t * K + k] * H + j);
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
            acc.x += a.x;
            acc.y += a.y;
            acc.z += b.x;
            acc.w += b.y;
        }
        *reinterpret_cast<float4*>(Y + (size_t)t * H + j) = acc;
    }
}

__global__ void k_err_to_status(const uint32_t* err, uint32_t* st) {
    if (threadIdx.x == 0 && *err) set_status(st, E0_ST_TIMEOUT);
}

// ------------------------------------------------------------------ host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Encoded tensor maps are kept, keyed by everything the encoding reads (the
// kind of map, base address and sizes), so that a call with the buffers of an
// earlier one skips the driver's encode: a cached map equals a fresh one.
struct MapKey {
    int kind;
    const void* base;
    uint64_t a, b, c, d;
    bool operator==(const MapKey& o) const {
        return kind == o.kind && base == o.base && a == o.a && b == o.b && c == o.c && d == o.d;
    }
};
struct MapEntry {
    MapKey key;
    CUtensorMap map;
};
static std::mutex g_map_mu;
static std::vector<MapEntry> g_maps;  // most recently added last
constexpr size_t MAP_CACHE = 64;

template <class Encode>
static bool cached_map(CUtensorMap* m, const MapKey& k, Encode encode) {
    {
        std::lock_guard<std::mutex> g(g_map_mu);
        for (const MapEntry& e : g_maps)
            if (e.key == k) {
                *m = e.map;
                return true;
            }
    }
    if (!encode(m)) return false;
    std::lock_guard<std::mutex> g(g_map_mu);
    if (g_maps.size() >= MAP_CACHE) g_maps.erase(g_maps.begin());
    g_maps.push_back(MapEntry{k, *m});
    return true;
}

// 2-D fp16 row-major [rows][inner] tensor, box = 64 elements x box_rows, 128B swizzle
static bool encode_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D uint8 [n_slots][rows][inner] view of one code region of every slot;
// box = 32 bytes x 128 rows x 1 slot, no swizzle (dense 32-byte rows).
static bool encode_codes_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t slots,
                             uint64_t slot_stride) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {inner, rows, slots};
    cuuint64_t strides[2] = {inner, slot_stride};
    cuuint32_t box[3] = {64, 128, 1};  // one K step of 128 inputs of 128 rows
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 5-D map over the down codes of every slot, in row blocks: {16 bytes, DROWS
// rows of a block, I/32 half-groups, H/DROWS blocks, slots}; one box = four
// half-groups (one 128-input K step) of 128 rows (8 blocks), stored
// [8][4][DROWS][16 B] in shared memory.
static bool encode_down_map(CUtensorMap* m, const void* base, uint64_t H, uint64_t I, uint64_t slots,
                            uint64_t slot_stride) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[5] = {16, DROWS, I / 32, H / DROWS, slots};
    cuuint64_t strides[4] = {16, (cuuint64_t)DROWS * 16, (I / 32) * DROWS * 16, slot_stride};
    cuuint32_t box[5] = {16, DROWS, 4, 128 / DROWS, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
    return cached_map(m, MapKey{0, base, inner, rows, box_rows, 0},
                      [&](CUtensorMap* o) { return encode_map(o, base, inner, rows, box_rows); });
}
static bool make_codes_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t slots,
                           uint64_t slot_stride) {
    return cached_map(m, MapKey{1, base, inner, rows, slots, slot_stride},
                      [&](CUtensorMap* o) { return encode_codes_map(o, base, inner, rows, slots, slot_stride); });
}
static bool make_down_map(CUtensorMap* m, const void* base, uint64_t H, uint64_t I, uint64_t slots,
                          uint64_t slot_stride) {
    return cached_map(m, MapKey{2, base, H, I, slots, slot_stride},
                      [&](CUtensorMap* o) { return encode_down_map(o, base, H, I, slots, slot_stride); });
}

static std::once_flag g_prefill_init;
static void prefill_attrs() {
    cudaFuncSetAttribute(k_router_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)router_gemm_smem());
    cudaFuncSetAttribute(k_umma2<MODE_GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemm2_smem());
    cudaFuncSetAttribute(k_umma2<MODE_DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemm2_smem());
}

int moe_prefill_forward(const uint16_t* Xu, int T, const e0_slot_pool* bank, const uint16_t* W_ru,
                        const e0_route_params* rpp, float* Y, int32_t* inds_out, float* w_out, void* ws,
                        uint32_t* st, cudaStream_t s) {
    std::call_once(g_prefill_init, prefill_attrs);
    const int H = bank->H, I = bank->I, E = bank->E, K = rpp->K;
    if (H % BM || I % BM) return E0_ERR_UNSUPPORTED;
    const __half* X = reinterpret_cast<const __half*>(Xu);
    const __half* W_r = reinterpret_cast<const __half*>(W_ru);
    PrefillWs w = prefill_ws(reinterpret_cast<char*>(ws), T, H, I, E, K);
    const int A = T * K;
    RouteP rp;
    rp.mode = rpp->mode;
    rp.K = K;
    rp.n_groups = rpp->n_groups > 0 ? rpp->n_groups : 1;
    rp.topk_groups = rpp->topk_groups > 0 ? rpp->topk_groups : 1;
    rp.scale = rpp->scale;
    rp.logit_bias = rpp->logit_bias;
    int32_t* inds = inds_out ? inds_out : w.inds;
    float* wts = w_out ? w_out : w.w;
    if (cudaMemsetAsync(w.err, 0, 4, s) != cudaSuccess) return E0_ERR_CUDA;

    CUtensorMap mWr, mX, mXp, mA;
    if (!make_map(&mWr, W_r, H, E, BM) || !make_map(&mX, X, H, T, BN) || !make_map(&mXp, w.xp, H, A, BN) ||
        !make_map(&mA, w.abuf, I, A, BN))
        return E0_ERR_CUDA;

    GemmP gp;
    memset(&gp, 0, sizeof(gp));
    gp.T = T;
    gp.E = E;
    gp.H = H;
    gp.I = I;
    gp.logits = w.logits;
    gp.pool = bank->data;
    gp.table = bank->slot_table;
    gp.n_slots = bank->n_slots;
    gp.slot_bytes = slot_bytes(H, I);
    gp.tiles = w.tiles;
    gp.n_tiles = w.n_tiles;
    gp.abuf = w.abuf;
    gp.yp = w.yp;
    gp.wp = w.wp;
    gp.perm = w.perm;
    gp.Y = Y;
    gp.Kr = K;
    // Y = sum_k w_k expert_k(x): by default the down epilogue adds each
    // weighted row into Y with fp32 atomics (the order of a token's K terms
    // varies from run to run); E0MOE_PREFILL_FIXED_ORDER=1 keeps fp16 rows and
    // sums them in a fixed order (identical bits on every run)
    const char* fo = getenv("E0MOE_PREFILL_FIXED_ORDER");
    gp.accumulate = (fo && atoi(fo) != 0) ? 0 : 1;
    gp.err = w.err;
    gp.st = st;

    // 1. router logits
    gp.K = H;
    gp.rows_out = E;
    k_router_gemm<<<dim3((E + BM - 1) / BM, (T + BN - 1) / BN), GEMM_THREADS, router_gemm_smem(), s>>>(
        mWr, mX, gp);
    // 2. routing (+ refinement of near-ties)
    int32_t* flag = w.flag;
    if (cudaMemsetAsync(flag, 0, 4, s) != cudaSuccess) return E0_ERR_CUDA;
    launch_route(false, w.logits, w.logits, X, H, W_r, T, E, rp, flag, w.done, inds, wts, st, s);
    launch_route(true, w.logits, w.logits, X, H, W_r, T, E, rp, flag, w.done, inds, wts, st, s);
    if (cudaGetLastError() != cudaSuccess) return E0_ERR_CUDA;
    // 3. sort
    int rc = sort_into(inds, T, K, E, w.counts, w.offsets, w.perm, w.pos, w, s);
    if (rc) return rc;
    k_prefill_tiles<<<1, 1024, 0, s>>>(w.counts, w.offsets, E, w.tiles, w.n_tiles);
    // 4. gather
    k_prefill_gather<<<A, 128, 0, s>>>(X, H, K, w.perm, wts, A, w.xp, w.wp);
    // 5. gate/up and 6. down: persistent grouped GEMMs, one CTA per SM
    CUtensorMap mGU, mDN;
    const size_t sbytes = slot_bytes(H, I);
    if (!make_codes_map(&mGU, bank->data, (uint64_t)H / 2, (uint64_t)2 * I, (uint64_t)bank->n_slots, sbytes) ||
        !make_down_map(&mDN, bank->data + SlotLayout{H, I}.down_codes(), (uint64_t)H, (uint64_t)I,
                       (uint64_t)bank->n_slots, sbytes))
        return E0_ERR_CUDA;
    gp.K = H;
    gp.rows_out = 2 * I;
    k_umma2<MODE_GATEUP><<<num_sms(), P2_THREADS, gemm2_smem(), s>>>(mGU, mXp, gp);
    gp.K = I;
    gp.rows_out = H;
    if (gp.accumulate && cudaMemsetAsync(Y, 0, (size_t)T * H * 4, s) != cudaSuccess) return E0_ERR_CUDA;
    k_umma2<MODE_DOWN><<<num_sms(), P2_THREADS, gemm2_smem(), s>>>(mDN, mA, gp);
    // 7. combine (fixed order only)
    if (!gp.accumulate) k_prefill_combine<<<T, 256, 0, s>>>(w.yp, w.pos, T, K, H, Y);
    // a GEMM that gave up waiting surfaces as E0_ST_TIMEOUT
    k_err_to_status<<<1, 32, 0, s>>>(w.err, st);
    if (cudaGetLastError() != cudaSuccess) return E0_ERR_CUDA;
    return E0_OK;
}

}  // namespace e0
