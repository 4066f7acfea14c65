// Decode-path device code: routing warps and the per-layer phases of the MoE
// block (router GEMV, gate/up, down), shared by the per-phase kernels and the
// persistent whole-token kernel.
//
// Work mapping used by every GEMV here: a row of n inputs is split into n/64
// groups; one lane owns one group (32 contiguous code bytes for int4, 128
// bytes for fp16), so a warp streams one row of a 2048-wide matrix as 1 KB
// (int4) of fully coalesced 16-byte loads.  Rows narrower than 32 groups are
// packed several to a warp (R = 32 / G rows per pass) and reduced with a
// segmented shuffle sum.
#pragma once
#include <math.h>

#include "e0_common.cuh"

namespace e0 {

// ------------------------------------------------------------------ parameters

struct RouteP {
    int32_t mode, K, n_groups, topk_groups;
    float scale;
    const float* logit_bias;
};

// One layer as the decode phases see it.
struct LayerP {
    const uint8_t* pool;      // slot data, kernel layout
    const int32_t* table;     // [E] expert -> slot
    int32_t n_slots;
    const __half* W_r;        // [E][H] router (may be null)
    // shared expert (sh == null: none)
    const uint8_t* sh;
    const __half *Ag, *Bg, *Au, *Bu, *Ad, *Bd;  // LoRA (Ag == null: none)
    int32_t rank;
    float lscale;             // alpha / rank
    // prerouter head owned by this layer (fc1 == null: none)
    const __half *fc1, *b1, *fc2, *b2, *lres;
    int32_t hidden;
    int32_t consumer;
};

struct DecodeArgs {
    int T, H, I, E, K;
    const float* x;           // [T][H] MoE input h
    const float* resid;       // [T][H] added to the output, or null
    const int32_t* inds;      // [T][K] routing used
    const float* w;           // [T][K]
    const int32_t* inds_prev; // [T][K] previous token's routing of this layer (head), or null
    LayerP L;
    float* a;                 // [T][K][I]
    float* gs;                // [T][I] shared gate (raw, before LoRA)
    float* us;                // [T][I]
    float* zg;                // [T][rank]  A_gate h
    float* zu;                // [T][rank]  A_up h
    float* hpre;              // [T][hidden] fc1 f + b1
    float* zres;              // [T][E]  lres f
    float* y;                 // [T][H]  output (may alias resid)
    float* z;                 // [T][E]  head logits, or null
    float* logits;            // [T][E]  router logits (router phase)
    uint32_t* st;
};

// ------------------------------------------------------------------ routing

// A float (not NaN) as an unsigned integer of the same order; -0 and +0 map
// alike.  0 is the key of no number (its inverse is a NaN pattern), so it
// stays free for "no candidate".
E0_DEV uint32_t float_order_key(float x) {
    uint32_t u = __float_as_uint(x);
    if ((u << 1) == 0) u = 0;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
E0_DEV float float_of_order_key(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// One warp routes one token.  Ranking uses the fp32 logits (softmax and
// sigmoid are monotonic), ties go to the lower expert id, output is in
// descending score order.  scr: E floats of per-warp shared scratch.
// With GAP the selection runs one round further and the function returns
// (the same in every lane) the smallest distance between consecutive ranked
// scores among the K + 1 largest (biased) logits, and, in group-limited
// routing, between the G-th and (G+1)-th group scores: a routing that a
// smaller logit error could change has a gap below that error.  Without GAP
// it returns +inf.
template <int MAXM, bool GAP = false>
E0_DEV float route_warp_t(const float* lg, int E, const RouteP& rp, int32_t* inds, float* w, float* scr,
                          uint32_t* st, int lane) {
    // scores are held as order keys (see float_order_key): ranking needs
    // only their order, and the winners' values are decoded from the keys
    uint32_t key[MAXM];
    bool bad = false;
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
        const int e = lane + 32 * m;
        float x = -INFINITY;
        if (e < E) {
            x = ld_shared_or_l2(lg + e) + (rp.logit_bias ? rp.logit_bias[e] : 0.f);
            if (!isfinite(x)) {
                bad = true;
                x = -INFINITY;
            }
        }
        key[m] = float_order_key(x);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(st, E0_ST_NONFINITE);
    uint32_t alive = 0;
#pragma unroll
    for (int m = 0; m < MAXM; ++m)
        if (lane + 32 * m < E) alive |= 1u << m;
    float gap = INFINITY;

    if (rp.mode == E0_ROUTE_SIGMOID_GROUP) {
        const int n = rp.n_groups, gsz = E / rp.n_groups;
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            const int e = lane + 32 * m;
            if (e < E) scr[e] = sigmoid_f(float_of_order_key(key[m]));
        }
        __syncwarp();
        float gscore = -INFINITY;
        if (lane < n) {
            float t1 = -1.f, t2 = -1.f;
            for (int j = 0; j < gsz; ++j) {
                const float s = scr[lane * gsz + j];
                if (s > t1) {
                    t2 = t1;
                    t1 = s;
                } else if (s > t2) {
                    t2 = s;
                }
            }
            gscore = gsz >= 2 ? t1 + t2 : t1;
        }
        __syncwarp();
        uint32_t kept = 0;
        float gv = gscore, gprev = 0.f;
        // with GAP, one more round finds the best group left out
        const int g_rounds = GAP ? min(rp.topk_groups + 1, n) : rp.topk_groups;
        for (int r = 0; r < g_rounds; ++r) {
            float bv = gv;
            int bi = lane < n ? lane : 64 + lane;
            if (lane < n && (kept >> lane & 1u)) {
                bv = -INFINITY;
                bi = 64 + lane;
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (GAP && r == rp.topk_groups) {
                if (bi < n) gap = fminf(gap, gprev - bv);
                break;
            }
            gprev = bv;
            if (bi < n) kept |= 1u << bi;
        }
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            const int e = lane + 32 * m;
            if (e < E && !((kept >> (e / gsz)) & 1u)) alive &= ~(1u << m);
        }
    }

    // Each round takes the largest live score with two warp reductions: the
    // largest order key (a float's order as an unsigned integer, 0 for "no
    // candidate"), then the lowest expert id holding it.
    int my_ind = -1;
    float my_val = 0.f, eprev = 0.f;
    for (int k = 0; k < (GAP ? rp.K + 1 : rp.K); ++k) {
        uint32_t bk = 0;
        uint32_t bi = 0xffffffffu;
#pragma unroll
        for (int m = 0; m < MAXM; ++m)
            if (((alive >> m) & 1u) && key[m] > bk) {  // strict: the lower id wins a tie
                bk = key[m];
                bi = (uint32_t)(lane + 32 * m);
            }
        const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
        if (mk == 0) break;  // fewer candidates than K (validated away on the host)
        const uint32_t wi = __reduce_min_sync(0xffffffffu, bk == mk ? bi : 0xffffffffu);
        if ((int)(wi & 31) == lane) alive &= ~(1u << (wi >> 5));
        if (GAP) {
            const float v = float_of_order_key(mk);
            if (k > 0) gap = fminf(gap, eprev - v);
            eprev = v;
            if (k == rp.K) break;
        }
        if (lane == k) {
            my_ind = (int)wi;
            my_val = float_of_order_key(mk);
        }
    }
    float wk;
    if (rp.mode == E0_ROUTE_SIGMOID_GROUP) {
        const float s = (lane < rp.K && my_ind >= 0) ? sigmoid_f(my_val) : 0.f;
        const float den = warp_sum(s) + 1e-20f;
        wk = rp.scale * s / den;
    } else {
        const float top = __shfl_sync(0xffffffffu, my_val, 0);
        const float ex = (lane < rp.K && my_ind >= 0) ? expf(my_val - top) : 0.f;
        const float den = warp_sum(ex);
        wk = ex / den;
    }
    if (lane < rp.K) {
        inds[lane] = my_ind;
        w[lane] = wk;
    }
    return gap;
}

static __device__ __noinline__ void route_warp(const float* lg, int E, const RouteP& rp, int32_t* inds, float* w, float* scr, uint32_t* st,
                       int lane) {
    if (E <= 32) route_warp_t<1>(lg, E, rp, inds, w, scr, st, lane);
    else if (E <= 64) route_warp_t<2>(lg, E, rp, inds, w, scr, st, lane);
    else if (E <= 128) route_warp_t<4>(lg, E, rp, inds, w, scr, st, lane);
    else if (E <= 256) route_warp_t<8>(lg, E, rp, inds, w, scr, st, lane);
    else if (E <= 512) route_warp_t<16>(lg, E, rp, inds, w, scr, st, lane);
    else route_warp_t<32>(lg, E, rp, inds, w, scr, st, lane);
}

// ------------------------------------------------------------------ helpers

E0_DEV int resolve_slot(const LayerP& L, int E, int e, uint32_t* st) {
    if (e < 0 || e >= E) {
        set_status(st, E0_ST_BAD_EXPERT);
        return -1;
    }
    const int s = L.table[e];
    if (s < 0 || s >= L.n_slots) {
        set_status(st, E0_ST_SLOT_MISS);
        return -1;
    }
    return s;
}

// fp16 row slice (64 halves) . fp32 x slice (64 floats)
E0_DEV float h64_dot(const __half* wrow, const float* x) {
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 wv = ldg_stream(wrow + 8 * c);
        const float4 x0 = *reinterpret_cast<const float4*>(x + 8 * c);
        const float4 x1 = *reinterpret_cast<const float4*>(x + 8 * c + 4);
        const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        acc += h8_dot(wv, xs);
    }
    return acc;
}

struct RowMap {
    int G, R, r, g;
    bool active;
    E0_DEV RowMap(int n_in, int lane) {
        G = n_in / GROUP;
        R = G >= 32 ? 1 : 32 / G;
        r = lane / G;
        g = lane % G;
        active = lane < R * G;
    }
};

// ------------------------------------------------------------------ smem sizes

struct GateUpSmem {
    size_t planes, xg, slots, total;
    __host__ __device__ GateUpSmem(int T, int H, int K) {
        const int G = H / GROUP;
        planes = 0;
        xg = planes + (size_t)T * G * 8 * sizeof(uint4);
        slots = xg + (size_t)T * G * sizeof(XGroup);
        total = slots + (size_t)T * K * sizeof(int);
        total = (total + 15) & ~(size_t)15;
    }
};

struct DownSmem {
    size_t planes, xg, slots, wts, asb, zd, hid, total;
    __host__ __device__ DownSmem(int T, int I, int K, bool sh, int rank, int hidden) {
        const int G = I / GROUP, NE = K + (sh ? 1 : 0);
        planes = 0;
        xg = planes + (size_t)T * NE * G * 8 * sizeof(uint4);
        slots = xg + (size_t)T * NE * G * sizeof(XGroup);
        wts = slots + (size_t)T * K * sizeof(int);
        asb = wts + (size_t)T * K * sizeof(float);
        asb = (asb + 15) & ~(size_t)15;
        zd = asb + (sh ? (size_t)T * I * sizeof(float) : 0);
        hid = zd + (sh ? (size_t)T * rank * sizeof(float) : 0);
        hid = (hid + 15) & ~(size_t)15;
        total = hid + (size_t)T * hidden * sizeof(float);
        total = (total + 15) & ~(size_t)15;
    }
};

// ------------------------------------------------------------------ router phase

// logits[t][e] = W_r[e] . x_t   (fp16 weights, fp32 activations and accumulation)
E0_DEV void phase_router(const DecodeArgs& A, int blk, int nblk) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const RowMap rm(A.H, lane);
    const int nrow = (A.E + rm.R - 1) / rm.R;
    const int total = A.T * nrow;
    for (int task = blk * nw + warp; task < total; task += nblk * nw) {
        const int t = task / nrow, e = (task % nrow) * rm.R + rm.r;
        float acc = 0.f;
        if (rm.active && e < A.E)
            acc = h64_dot(A.L.W_r + (size_t)e * A.H + GROUP * rm.g, A.x + (size_t)t * A.H + GROUP * rm.g);
        acc = seg_sum(acc, rm.G, lane);
        if (rm.active && rm.g == 0 && e < A.E) A.logits[t * A.E + e] = acc;
    }
}

// ------------------------------------------------------------------ gate/up phase
//
// Tasks: routed row pairs (gate i, up i) of every (token, k); the shared
// expert's row pairs; the LoRA A projections of the shared gate and up; the
// head's fc1 rows and linear-residual rows.  `inds` may point to shared memory.
E0_DEV void phase_gateup(const DecodeArgs& A, const int32_t* inds, int blk, int nblk, char* smem) {
    const int T = A.T, H = A.H, I = A.I, K = A.K, E = A.E;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const GateUpSmem lay(T, H, K);
    uint4* planes = reinterpret_cast<uint4*>(smem + lay.planes);
    XGroup* xg = reinterpret_cast<XGroup*>(smem + lay.xg);
    int* slots = reinterpret_cast<int*>(smem + lay.slots);
    const int GH = H / GROUP;

    const bool have_pool = A.L.pool != nullptr;
    const bool need_planes = have_pool || A.L.sh != nullptr;
    if (need_planes)
        for (int q = warp; q < T * GH; q += nw)
            quantize_group_warp(A.x + (size_t)(q / GH) * H + GROUP * (q % GH), planes + q * 8, xg + q, lane, A.st);
    if (have_pool)
        for (int q = threadIdx.x; q < T * K; q += blockDim.x)
            slots[q] = resolve_slot(A.L, E, inds[q], blk == 0 ? A.st : nullptr);
    __syncthreads();

    const RowMap rm(H, lane);
    const int R = rm.R;
    const int nI = (I + R - 1) / R;
    const int n_routed = have_pool ? T * K * nI : 0;
    const int n_shared = A.L.sh ? T * nI : 0;
    const int nr = (A.L.rank + R - 1) / R;
    const int n_lora = (A.L.sh && A.L.Ag) ? T * 2 * nr : 0;
    const int nh = A.L.fc1 ? (A.L.hidden + R - 1) / R : 0;
    const int ne = A.L.fc1 ? (E + R - 1) / R : 0;
    const int n_fc1 = T * nh, n_lres = T * ne;
    const int total = n_routed + n_shared + n_lora + n_fc1 + n_lres;
    const size_t sbytes = SlotLayout{H, I}.bytes();
    const size_t gu_sb = SlotLayout{H, I}.gu_sb();

    for (int task = blk * nw + warp; task < total; task += nblk * nw) {
        if (task < n_routed + n_shared) {
            int t, k, i;
            const uint8_t* ex;
            bool routed = task < n_routed;
            if (routed) {
                t = task / (K * nI);
                const int rem = task % (K * nI);
                k = rem / nI;
                i = (rem % nI) * R + rm.r;
                const int s = slots[t * K + k];
                ex = s >= 0 ? A.L.pool + (size_t)s * sbytes : nullptr;
            } else {
                const int q = task - n_routed;
                t = q / nI;
                k = 0;
                i = (q % nI) * R + rm.r;
                ex = A.L.sh;
            }
            float pg = 0.f, pu = 0.f;
            const bool live = rm.active && i < I && ex != nullptr;
            if (live) {
                const uint8_t* gp = ex + (size_t)i * H + 32 * rm.g;
                const uint4 g0 = ldg_stream(gp), g1 = ldg_stream(gp + 16);
                const uint4 u0 = ldg_stream(gp + H / 2), u1 = ldg_stream(gp + H / 2 + 16);
                const uint32_t sbg = ldg_u32(ex + gu_sb + ((size_t)(2 * i) * GH + rm.g) * 4);
                const uint32_t sbu = ldg_u32(ex + gu_sb + ((size_t)(2 * i + 1) * GH + rm.g) * 4);
                const int pq = t * GH + rm.g;
                pg = q4_group_dot(g0, g1, planes + pq * 8, xg[pq], sbg);
                pu = q4_group_dot(u0, u1, planes + pq * 8, xg[pq], sbu);
            }
            pg = seg_sum(pg, rm.G, lane);
            pu = seg_sum(pu, rm.G, lane);
            if (rm.active && rm.g == 0 && i < I) {
                if (routed) {
                    A.a[((size_t)t * K + k) * I + i] = ex ? silu_f(pg) * pu : 0.f;
                } else {
                    A.gs[(size_t)t * I + i] = pg;
                    A.us[(size_t)t * I + i] = pu;
                }
            }
            continue;
        }
        int q = task - n_routed - n_shared;
        if (q < n_lora) {
            // z_g / z_u = A_gate h, A_up h  (fp16 rows of H inputs)
            const int t = q / (2 * nr), which = (q / nr) % 2, rr = (q % nr) * R + rm.r;
            const __half* Am = which ? A.L.Au : A.L.Ag;
            float acc = 0.f;
            if (rm.active && rr < A.L.rank)
                acc = h64_dot(Am + (size_t)rr * H + GROUP * rm.g, A.x + (size_t)t * H + GROUP * rm.g);
            acc = seg_sum(acc, rm.G, lane);
            if (rm.active && rm.g == 0 && rr < A.L.rank) (which ? A.zu : A.zg)[t * A.L.rank + rr] = acc;
            continue;
        }
        q -= n_lora;
        // head rows: fc1 (hidden rows) then lres (E rows), each H + 2E wide
        const bool is_fc1 = q < n_fc1;
        if (!is_fc1) q -= n_fc1;
        const int per = is_fc1 ? nh : ne;
        const int t = q / per, row = (q % per) * R + rm.r;
        const int nrows = is_fc1 ? A.L.hidden : E;
        const __half* Wm = is_fc1 ? A.L.fc1 : A.L.lres;
        const size_t ld = (size_t)H + 2 * E;
        float acc = 0.f;
        if (rm.active && row < nrows) {
            const __half* wr = Wm + (size_t)row * ld;
            acc = h64_dot(wr + GROUP * rm.g, A.x + (size_t)t * H + GROUP * rm.g);
            // the one-hot blocks: only the 2K routed columns are read
            for (int c = rm.g; c < 2 * K; c += rm.G) {
                int e;
                size_t col;
                if (c < K) {
                    e = inds[t * K + c];
                    col = (size_t)H + e;
                } else {
                    e = A.inds_prev ? A.inds_prev[t * K + c - K] : -1;
                    col = (size_t)H + E + e;
                }
                if (e >= 0 && e < E) acc += __half2float(wr[col]);
            }
        }
        acc = seg_sum(acc, rm.G, lane);
        if (rm.active && rm.g == 0 && row < nrows) {
            if (is_fc1) A.hpre[(size_t)t * A.L.hidden + row] = acc + (A.L.b1 ? __half2float(A.L.b1[row]) : 0.f);
            else A.zres[(size_t)t * E + row] = acc;
        }
    }
}

// ------------------------------------------------------------------ down phase
//
// y[t][j] = resid + sum_k w_k D_k[j] . a_k + D_s[j] . a_s + (alpha/r) B_d[j] . (A_d a_s)
// and the head's second layer z[t][e] = fc2[e] . gelu(hpre_t) + b2[e] + zres[t][e].
E0_DEV void phase_down(const DecodeArgs& A, int blk, int nblk, char* smem) {
    const int T = A.T, H = A.H, I = A.I, K = A.K, E = A.E;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const bool sh = A.L.sh != nullptr;
    const bool lora = sh && A.L.Ag != nullptr;
    const bool head = A.L.fc1 != nullptr && A.z != nullptr;
    const int rank = lora ? A.L.rank : 0;
    const int hidden = head ? A.L.hidden : 0;
    const DownSmem lay(T, I, A.L.pool != nullptr ? K : 0, sh, rank, hidden);
    uint4* planes = reinterpret_cast<uint4*>(smem + lay.planes);
    XGroup* xg = reinterpret_cast<XGroup*>(smem + lay.xg);
    int* slots = reinterpret_cast<int*>(smem + lay.slots);
    float* wts = reinterpret_cast<float*>(smem + lay.wts);
    float* asb = reinterpret_cast<float*>(smem + lay.asb);
    float* zd = reinterpret_cast<float*>(smem + lay.zd);
    float* hid = reinterpret_cast<float*>(smem + lay.hid);
    const bool have_pool = A.L.pool != nullptr;
    const int NK = have_pool ? K : 0;
    const int GI = I / GROUP, NE = NK + (sh ? 1 : 0);

    for (int q = threadIdx.x; q < T * NK; q += blockDim.x) {
        slots[q] = resolve_slot(A.L, E, ldi_shared_or_l2(A.inds + q), nullptr);
        wts[q] = ld_shared_or_l2(A.w + q);
    }
    if (sh) {
        for (int q = threadIdx.x; q < T * I; q += blockDim.x) {
            const int t = q / I, i = q % I;
            float g = __ldcg(A.gs + q), u = __ldcg(A.us + q);
            if (lora) {
                float dg = 0.f, du = 0.f;
                for (int rr = 0; rr < rank; ++rr) {
                    dg = fmaf(__half2float(A.L.Bg[(size_t)i * rank + rr]), __ldcg(A.zg + t * rank + rr), dg);
                    du = fmaf(__half2float(A.L.Bu[(size_t)i * rank + rr]), __ldcg(A.zu + t * rank + rr), du);
                }
                g = fmaf(A.L.lscale, dg, g);
                u = fmaf(A.L.lscale, du, u);
            }
            asb[q] = silu_f(g) * u;
        }
    }
    if (head)
        for (int q = threadIdx.x; q < T * hidden; q += blockDim.x) hid[q] = gelu_erf_f(__ldcg(A.hpre + q));
    __syncthreads();
    for (int q = warp; q < T * NE * GI; q += nw) {
        const int t = q / (NE * GI), rem = q % (NE * GI), k = rem / GI, g = rem % GI;
        const float* src = k < NK ? A.a + ((size_t)t * K + k) * I + GROUP * g : asb + (size_t)t * I + GROUP * g;
        quantize_group_warp(src, planes + q * 8, xg + q, lane, A.st);
    }
    if (lora) {
        for (int q = warp; q < T * rank; q += nw) {
            const int t = q / rank, rr = q % rank;
            float acc = 0.f;
            for (int i = lane; i < I; i += 32)
                acc = fmaf(__half2float(A.L.Ad[(size_t)rr * I + i]), asb[(size_t)t * I + i], acc);
            acc = warp_sum(acc);
            if (lane == 0) zd[q] = acc;
        }
    }
    __syncthreads();

    const RowMap rm(I, lane);
    const int R = rm.R;
    const int nj = (H + R - 1) / R;
    const int n_down = (have_pool || sh) ? T * nj : 0;
    const RowMap rh(head ? hidden : GROUP, lane);
    const int ner = head ? (E + rh.R - 1) / rh.R : 0;
    const int n_fc2 = T * ner;
    const SlotLayout sl{H, I};
    const size_t sbytes = sl.bytes();

    for (int task = blk * nw + warp; task < n_down + n_fc2; task += nblk * nw) {
        if (task < n_down) {
            const int t = task / nj, j = (task % nj) * R + rm.r;
            float acc = 0.f;
            const bool live = rm.active && j < H;
            if (live) {
                for (int k = 0; k < NK; ++k) {
                    const int s = slots[t * K + k];
                    if (s < 0) continue;
                    const uint8_t* ex = A.L.pool + (size_t)s * sbytes;
                    const uint8_t* cp = ex + sl.down_code_off(j, 2 * rm.g);
                    const uint4 c0 = ldg_stream(cp), c1 = ldg_stream(cp + (size_t)DROWS * 16);
                    const uint32_t sb = ldg_u32(ex + sl.down_sb_off(j, rm.g));
                    const int pq = (t * NE + k) * GI + rm.g;
                    acc = fmaf(wts[t * K + k], q4_group_dot(c0, c1, planes + pq * 8, xg[pq], sb), acc);
                }
                if (sh) {
                    const uint8_t* cp = A.L.sh + sl.down_code_off(j, 2 * rm.g);
                    const uint4 c0 = ldg_stream(cp), c1 = ldg_stream(cp + (size_t)DROWS * 16);
                    const uint32_t sb = ldg_u32(A.L.sh + sl.down_sb_off(j, rm.g));
                    const int pq = (t * NE + NK) * GI + rm.g;
                    acc += q4_group_dot(c0, c1, planes + pq * 8, xg[pq], sb);
                }
            }
            acc = seg_sum(acc, rm.G, lane);
            if (live && rm.g == 0) {
                if (lora) {
                    float d = 0.f;
                    for (int rr = 0; rr < rank; ++rr)
                        d = fmaf(__half2float(A.L.Bd[(size_t)j * rank + rr]), zd[t * rank + rr], d);
                    acc = fmaf(A.L.lscale, d, acc);
                }
                if (A.resid) acc += ld_shared_or_l2(A.resid + (size_t)t * H + j);
                A.y[(size_t)t * H + j] = acc;
            }
        } else {
            const int q = task - n_down;
            const int t = q / ner, e = (q % ner) * rh.R + rh.r;
            float acc = 0.f;
            if (rh.active && e < E)
                acc = h64_dot(A.L.fc2 + (size_t)e * hidden + GROUP * rh.g, hid + (size_t)t * hidden + GROUP * rh.g);
            acc = seg_sum(acc, rh.G, lane);
            if (rh.active && rh.g == 0 && e < E)
                A.z[(size_t)t * E + e] = acc + (A.L.b2 ? __half2float(A.L.b2[e]) : 0.f) + __ldcg(A.zres + (size_t)t * E + e);
        }
    }
}

// h = r / sqrt(mean(r^2) + eps) for one row, by one block (blockDim multiple of 32).
E0_DEV void rmsnorm_block(const float* r, float* h, int H, float eps, float* red /*32 floats smem*/) {
    float s = 0.f;
    for (int j = threadIdx.x; j < H; j += blockDim.x) s = fmaf(r[j], r[j], s);
    s = warp_sum(s);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = s;
    __syncthreads();
    if (warp == 0) {
        float v = lane < nw ? red[lane] : 0.f;
        v = warp_sum(v);
        if (lane == 0) red[0] = v;
    }
    __syncthreads();
    const float denom = sqrtf(red[0] / (float)H + eps);
    for (int j = threadIdx.x; j < H; j += blockDim.x) h[j] = r[j] / denom;
    __syncthreads();
}

}  // namespace e0
