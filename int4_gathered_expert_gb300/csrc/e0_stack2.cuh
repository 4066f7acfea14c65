// One decode token over all layers in one launch, one grid barrier per layer.
//
// The launch is made of teams: thread-block clusters of TEAM CTAs (one CTA
// per SM).  Each layer's expert work — the K routed experts plus the shared
// expert — is cut into half-groups of 32 intermediate rows; every team takes
// a contiguous run of half-groups.  Inside a team each CTA computes a slice
// of the SwiGLU activations a = silu(G h) * (U h) for the team's rows and
// writes them into every team member's shared memory (distributed shared
// memory), one cluster barrier later every member holds the team's
// activations, quantises them, and computes the partial down projection
// sum_k w_k D_k[:, team columns] a_k for its share of the output rows.  The
// partial sums are added into the layer output y with red.add; the grid
// barrier at the end of the layer is the only grid-wide synchronisation
// (native-routing layers add one for the router logits).
//
// Every CTA keeps the residual stream r in its own shared memory and
// updates it from y at the start of the next layer, so the RMSNorm needs one
// 8 KB read per CTA and no extra barrier.  The prerouter head runs on four
// auxiliary warps per CTA alongside the expert warps: fc1 and the linear
// residual of the owner layer l, fc2 of owner l-1 (its hidden vector is
// complete once layer l starts), and the routing of owner l-2's logits.
// Weights of layer l+1 are prefetched into L2 at the start of layer l; for
// consumer layers the routed experts are known one token ahead (prediction
// as routing), so their bytes are in flight long before they are used.
// Included inside namespace e0 of e0_decode.cu (it uses StackHdr and the
// phase helpers defined there).
#pragma once

constexpr int TEAM = 8;             // CTAs per cluster
constexpr int T2_THREADS = 384;     // 12 warps
constexpr int T2_EXPERT_WARPS = 12; // warps 0..11: experts; 12..15: head and bookkeeping
constexpr int T2_MAX_UNITS = 32;    // half-groups per team
constexpr int T2_MAX_RANK = 64;

// ------------------------------------------------------------------ cluster primitives

E0_DEV uint32_t cl_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
E0_DEV uint32_t cl_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
E0_DEV uint32_t cl_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
E0_DEV void cl_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
E0_DEV void cl_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
E0_DEV void cl_sync() {
    cl_arrive();
    cl_wait();
}
E0_DEV uint32_t cl_map(const void* local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(r)
                 : "r"((uint32_t)__cvta_generic_to_shared(local)), "r"(rank));
    return r;
}
E0_DEV void cl_st(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

E0_DEV void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// This CTA's 1/n share of a byte range, prefetched into L2.
E0_DEV void prefetch_share(const void* base, size_t bytes, int b, int n) {
    if (!base || bytes < 16) return;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(base) & ~(uintptr_t)15;
    const uintptr_t a1 = (reinterpret_cast<uintptr_t>(base) + bytes + 15) & ~(uintptr_t)15;
    const size_t total = a1 - a0;
    size_t chunk = (total / n + 15) & ~(size_t)15;
    if (chunk < 256) chunk = 256;
    const size_t s0 = (size_t)b * chunk;
    if (s0 >= total) return;
    size_t len = total - s0 < chunk ? total - s0 : chunk;
    for (size_t o = 0; o < len; o += 65536) {
        const size_t piece = len - o < 65536 ? len - o : 65536;
        prefetch_l2(reinterpret_cast<const void*>(a0 + s0 + o), (uint32_t)piece);
    }
}

// ------------------------------------------------------------------ barrier

// Grid barrier on a 64-bit monotonic counter: arrive with a release add,
// wait with acquire loads until the counter reaches the target; gives up
// after a bounded number of polls (or when another CTA already did),
// raising E0_ST_TIMEOUT.
E0_DEV void grid_barrier2(StackHdr* S, unsigned long long target, uint32_t* st) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(&S->bar_ctr), "l"(1ull) : "memory");
        uint32_t it = 0;
        while (true) {
            unsigned long long v;
            asm volatile("ld.acquire.gpu.u64 %0, [%1];" : "=l"(v) : "l"(&S->bar_ctr) : "memory");
            if (v >= target) break;
            unsigned ab;
            asm volatile("ld.relaxed.gpu.u32 %0, [%1];" : "=r"(ab) : "l"(&S->bar_abort) : "memory");
            if (ab) break;
            if (++it > (1u << 24)) {
                set_status(st, E0_ST_TIMEOUT);
                atomicExch(&S->bar_abort, 1u);
                break;
            }
        }
    }
    __syncthreads();
}

// ------------------------------------------------------------------ quantise / dot (32-element half-groups)

// One warp quantises 32 values (one per lane; lanes beyond n hold 0) into
// the planes of a half-group (4 uint4, kernel nibble order) and its XGroup.
E0_DEV void quantize_half_warp(float v, uint4* planes, XGroup* xg, int lane) {
    const float mx = warp_max(fabsf(v));
    const float inv = (mx > 0.f && mx < 3.0e38f) ? 32767.f / mx : 0.f;
    int q = __float2int_rn(v * inv);
    q = max(-32767, min(32767, q));
    const int s = warp_sum_int(q);
    const int e = lane & 7;  // element within its 8-element word
    const int set = (e >> 1) & 1, byte = ((e & 1) << 1) | (e >> 2);
    const uint32_t hi = ((uint32_t)(q >> 8) & 0xFFu) << (8 * byte);
    const uint32_t lo = ((uint32_t)q & 0xFFu) << (8 * byte);
    uint32_t hiA = set ? 0u : hi, hiB = set ? hi : 0u, loA = set ? 0u : lo, loB = set ? lo : 0u;
#pragma unroll
    for (int o = 1; o <= 4; o <<= 1) {
        hiA |= __shfl_xor_sync(0xffffffffu, hiA, o);
        hiB |= __shfl_xor_sync(0xffffffffu, hiB, o);
        loA |= __shfl_xor_sync(0xffffffffu, loA, o);
        loB |= __shfl_xor_sync(0xffffffffu, loB, o);
    }
    if (e == 0) planes[lane >> 3] = make_uint4(hiA, hiB, loA, loB);
    if (lane == 0) {
        xg->c = (inv > 0.f) ? mx / 32767.f : 0.f;
        xg->sx = (float)s;
    }
}

// Dot product of one half-group of an int4 row (16 code bytes) with its planes.
E0_DEV float q4_half_dot(const uint4 c, const uint4* pl, XGroup xg, uint32_t sb_bits) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    int hi = 0;
    uint32_t lo = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint4 p = pl[k];
        const uint32_t a = w[k] & 0x0F0F0F0Fu;
        const uint32_t b = (w[k] >> 4) & 0x0F0F0F0Fu;
        hi = dp4a_us(a, p.x, hi);
        hi = dp4a_us(b, p.y, hi);
        lo = dp4a_uu(a, p.z, lo);
        lo = dp4a_uu(b, p.w, lo);
    }
    const int sqx = hi * 256 + (int)lo;
    __half2 sb = *reinterpret_cast<const __half2*>(&sb_bits);
    return xg.c * fmaf(__low2float(sb), (float)sqx, __high2float(sb) * xg.sx);
}

// ------------------------------------------------------------------ fp16 rows, one warp per row

E0_DEV float h8_dot44(const uint4 wv, const float4 a, const float4 b) {
    const __half2* hw = reinterpret_cast<const __half2*>(&wv);
    const float2 w0 = __half22float2(hw[0]), w1 = __half22float2(hw[1]);
    const float2 w2 = __half22float2(hw[2]), w3 = __half22float2(hw[3]);
    float acc = w0.x * a.x;
    acc = fmaf(w0.y, a.y, acc);
    acc = fmaf(w1.x, a.z, acc);
    acc = fmaf(w1.y, a.w, acc);
    acc = fmaf(w2.x, b.x, acc);
    acc = fmaf(w2.y, b.y, acc);
    acc = fmaf(w3.x, b.z, acc);
    return fmaf(w3.y, b.w, acc);
}

// This lane's part of an fp16 row (n halves, n a multiple of 8) times an fp32
// vector in shared memory: the lane takes 8 consecutive elements out of every
// 256, so one load of the warp covers 512 contiguous bytes of the row and the
// shared-memory reads of neighbouring lanes do not collide.  Sum the lanes
// with warp_sum.
__device__ __noinline__ float hrow_dot(const __half* w, const float* x, int n, int lane) {
    float acc = 0.f;
    for (int c0 = 0; c0 < n; c0 += 4 * 256) {
        uint4 wv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int c = c0 + k * 256 + lane * 8;
            if (c < n) wv[k] = ldg_stream(w + c);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int c = c0 + k * 256 + lane * 8;
            if (c < n)
                acc += h8_dot44(wv[k], *reinterpret_cast<const float4*>(x + c), *reinterpret_cast<const float4*>(x + c + 4));
        }
    }
    return acc;
}

// Same for the head's second layer: x = gelu_erf(hp), hp written by other
// blocks earlier in the launch (read from L2).
__device__ __noinline__ float hrow_dot_gelu(const __half* w, const float* hp, int n, int lane) {
    float acc = 0.f;
    for (int c0 = 0; c0 < n; c0 += 2 * 256) {
        uint4 wv[2];
        float4 a[2], b[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int c = c0 + k * 256 + lane * 8;
            if (c < n) {
                wv[k] = ldg_stream(w + c);
                a[k] = __ldcg(reinterpret_cast<const float4*>(hp + c));
                b[k] = __ldcg(reinterpret_cast<const float4*>(hp + c + 4));
            }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int c = c0 + k * 256 + lane * 8;
            if (c < n) {
                const float4 ga = make_float4(gelu_erf_f(a[k].x), gelu_erf_f(a[k].y), gelu_erf_f(a[k].z), gelu_erf_f(a[k].w));
                const float4 gb = make_float4(gelu_erf_f(b[k].x), gelu_erf_f(b[k].y), gelu_erf_f(b[k].z), gelu_erf_f(b[k].w));
                acc += h8_dot44(wv[k], ga, gb);
            }
        }
    }
    return acc;
}

// ------------------------------------------------------------------ shared memory layout

struct T2Smem {
    size_t r, h, hpl, hxg, ateam, apl, axg, zred, zg, zu, zd, inds, w, slots, scr, red, total;
    __host__ __device__ T2Smem(int H, int E, int L, int K) {
        const int GH = H / GROUP;
        const int max_rows = T2_MAX_UNITS * 32;
        size_t o = 0;
        r = o;
        o += (size_t)H * 4;
        h = o;
        o += (size_t)H * 4;
        hpl = o;
        o += (size_t)GH * 8 * 16;
        hxg = o;
        o += (size_t)GH * sizeof(XGroup);
        o = (o + 15) & ~(size_t)15;
        ateam = o;
        o += (size_t)max_rows * 4;
        apl = o;
        o += (size_t)T2_MAX_UNITS * 4 * 16;
        axg = o;
        o += (size_t)T2_MAX_UNITS * sizeof(XGroup);
        zred = o;
        o += (size_t)TEAM * 2 * T2_MAX_RANK * 4;
        zg = o;
        o += T2_MAX_RANK * 4;
        zu = o;
        o += T2_MAX_RANK * 4;
        zd = o;
        o += T2_MAX_RANK * 4;
        inds = o;  // [L][K] routing of every layer at this token
        o += (size_t)L * K * 4;
        w = o;
        o += (size_t)L * K * 4;
        o = (o + 15) & ~(size_t)15;
        slots = o;  // [L][K+1] expert data pointers (last: shared expert)
        o += (size_t)L * (K + 1) * 8;
        scr = o;
        o += (size_t)2 * E * 4;
        red = o;
        o += 32 * 4;
        total = (o + 127) & ~(size_t)127;
    }
};

// Work split of one layer: NU half-group units (routed experts first, then the
// shared expert), team tau of NT takes units [u0, u1).
struct T2Split {
    int HG, NU, u0, u1, rows;
    E0_DEV T2Split(int I, int nk, int tau, int NT) {
        HG = I / 32;
        NU = nk * HG;
        u0 = (int)((long)tau * NU / NT);
        u1 = (int)((long)(tau + 1) * NU / NT);
        rows = (u1 - u0) * 32;
    }
};

E0_DEV void prefetch_line(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// This CTA's share (1/n) of a byte range, prefetched into L2 one 128-byte
// line per thread and step.
E0_DEV void prefetch_share_lines(const void* base, size_t bytes, int b, int n) {
    if (!base || bytes == 0) return;
    const size_t lines = (bytes + 127) / 128;
    const size_t per = (lines + n - 1) / n;
    const size_t l0 = (size_t)b * per, l1 = l0 + per < lines ? l0 + per : lines;
    const char* c = reinterpret_cast<const char*>(base);
    for (size_t q = l0 + threadIdx.x; q < l1; q += T2_THREADS) prefetch_line(c + q * 128);
}

// ------------------------------------------------------------------ the kernel

__global__ void __launch_bounds__(T2_THREADS, 1)
    k_stack_token2(StackHdr* Sp, const float* x, float* r_out, TraceP tr, uint32_t* st) {
    extern __shared__ __align__(16) char smem[];
    StackHdr& S = *Sp;
    const int H = S.H, I = S.I, E = S.E, K = S.K, Lz = S.L;
    const int GH = H / GROUP;
    const int t = S.t;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NW = T2_THREADS >> 5;
    const int nb = gridDim.x, b = blockIdx.x;
    const int team = (int)cl_id(), NT = (int)cl_count(), crank = (int)cl_rank();
    const unsigned long long bar0 = S.bar_base;
    int nbar = 0;

    const T2Smem lay(H, E, Lz, K);
    float* r = reinterpret_cast<float*>(smem + lay.r);
    float* h = reinterpret_cast<float*>(smem + lay.h);
    uint4* hpl = reinterpret_cast<uint4*>(smem + lay.hpl);
    XGroup* hxg = reinterpret_cast<XGroup*>(smem + lay.hxg);
    float* ateam = reinterpret_cast<float*>(smem + lay.ateam);
    uint4* apl = reinterpret_cast<uint4*>(smem + lay.apl);
    XGroup* axg = reinterpret_cast<XGroup*>(smem + lay.axg);
    float* zred = reinterpret_cast<float*>(smem + lay.zred);
    float* zg = reinterpret_cast<float*>(smem + lay.zg);
    float* zu = reinterpret_cast<float*>(smem + lay.zu);
    float* zd = reinterpret_cast<float*>(smem + lay.zd);
    int32_t* inds_all = reinterpret_cast<int32_t*>(smem + lay.inds);
    float* w_all = reinterpret_cast<float*>(smem + lay.w);
    const uint8_t** slot_all = reinterpret_cast<const uint8_t**>(smem + lay.slots);
    float* scr = reinterpret_cast<float*>(smem + lay.scr);
    float* red = reinterpret_cast<float*>(smem + lay.red);

    const SlotLayout sl{H, I};
    const size_t sbytes = sl.bytes();

    // ---- routing of every layer that takes a prediction this token (known now)
    for (int q = tid; q < Lz * (K + 1); q += T2_THREADS) {
        const int l = q / (K + 1), k = q % (K + 1);
        const LayerP& L = S.layers[l];
        if (k == K) {
            slot_all[q] = L.sh;
            continue;
        }
        if (layer_native(S, L, t)) continue;
        const size_t o = ((size_t)(t & 1) * Lz + l) * K + k;
        const int e = __ldcg(S.pred_inds + o);
        inds_all[l * K + k] = e;
        w_all[l * K + k] = __ldcg(S.pred_w + o);
        const int s2 = (e >= 0 && e < E) ? L.table[e] : -1;
        slot_all[q] = (s2 >= 0 && s2 < L.n_slots) ? L.pool + (size_t)s2 * sbytes : nullptr;
    }
    __syncthreads();

    for (int l = 0; l < Lz; ++l) {
        const LayerP L = S.layers[l];
        const bool native = layer_native(S, L, t);
        const bool sh = L.sh != nullptr;
        const bool lora = sh && L.Ag != nullptr;
        const int rank = lora ? L.rank : 0;
        const int nk = K + (sh ? 1 : 0);
        int32_t* inds_s = inds_all + l * K;
        float* w_s = w_all + l * K;
        const uint8_t** slot_s = slot_all + l * (K + 1);

        // ---- residual stream: r_l = x (l = 0) or r_{l-1} + y_{l-1}; h = RMSNorm(r)
        {
            const float* ysrc = l == 0 ? x : S.y_acc + (size_t)((l - 1) % 3) * H;
            float ss = 0.f;
            for (int j = tid * 4; j < H; j += T2_THREADS * 4) {
                const float4 y4 = __ldcg(reinterpret_cast<const float4*>(ysrc + j));
                float4 v;
                if (l == 0) {
                    v = y4;
                } else {
                    const float4 r4 = *reinterpret_cast<const float4*>(r + j);
                    v = make_float4(r4.x + y4.x, r4.y + y4.y, r4.z + y4.z, r4.w + y4.w);
                }
                *reinterpret_cast<float4*>(r + j) = v;
                ss = fmaf(v.x, v.x, ss);
                ss = fmaf(v.y, v.y, ss);
                ss = fmaf(v.z, v.z, ss);
                ss = fmaf(v.w, v.w, ss);
            }
            ss = warp_sum(ss);
            if (lane == 0) red[warp] = ss;
            __syncthreads();
            float tot = lane < NW ? red[lane] : 0.f;
            tot = warp_sum(tot);
            const float denom = sqrtf(tot / (float)H + 1e-6f);
            for (int j = tid; j < H; j += T2_THREADS) h[j] = r[j] / denom;
            if (b == 0 && tr.r)
                for (int j = tid; j < H; j += T2_THREADS) tr.r[(size_t)l * H + j] = r[j];
            // the output buffer of layer l+1 starts at zero
            if (b == nb - 1)
                for (int j = tid; j < H; j += T2_THREADS) S.y_acc[(size_t)((l + 1) % 3) * H + j] = 0.f;
        }
        __syncthreads();

        // ---- routing of native layers: logits on every warp of the grid, one grid barrier
        if (native) {
            for (int e = b * NW + warp; e < E; e += nb * NW) {
                const float acc = warp_sum(hrow_dot(L.W_r + (size_t)e * H, h, H, lane));
                if (lane == 0) S.logits[e] = acc;
            }
            grid_barrier2(Sp, bar0 + (unsigned long long)(++nbar) * nb, st);
            if (warp == 0) {
                stack_resolve(S, L, l, t, inds_s, w_s, scr, b == 0 ? st : nullptr, lane);
                if (lane < K) {
                    const int e = inds_s[lane];
                    const int s2 = (e >= 0 && e < E) ? L.table[e] : -1;
                    slot_s[lane] = (s2 >= 0 && s2 < L.n_slots) ? L.pool + (size_t)s2 * sbytes : nullptr;
                }
            }
            __syncthreads();  // warp 0's routing is read by every warp below
        }
        if (b == 0 && warp == 1 && lane < K) {
            const int e = inds_s[lane];
            if (!slot_s[lane]) set_status(st, (e < 0 || e >= E) ? E0_ST_BAD_EXPERT : E0_ST_SLOT_MISS);
            S.hist[((size_t)(t & 1) * Lz + l) * K + lane] = e;
            S.wcur[(size_t)l * K + lane] = w_s[lane];
            if (tr.inds) tr.inds[(size_t)l * K + lane] = e;
            if (tr.w) tr.w[(size_t)l * K + lane] = w_s[lane];
        }
        // planes of h: word k of group g sits at hpl[k * GH + g], so lanes that
        // read consecutive groups touch consecutive 16-byte words
        for (int g = warp; g < GH; g += NW) quantize_group_warp(h + GROUP * g, hpl + g, hxg + g, lane, nullptr, GH);
        __syncthreads();

        const T2Split sp(I, nk, team, NT);
        const int p0 = (int)((long)crank * sp.rows / TEAM), p1 = (int)((long)(crank + 1) * sp.rows / TEAM);
        const bool team_lora = lora && sp.u1 > K * sp.HG;

        // ---- LoRA A of the shared expert (teams holding shared rows): each
        // member reduces 1/TEAM of the inputs, partial sums exchanged
        if (team_lora) {
            const int c0 = crank * (H / TEAM), nc = H / TEAM;
            for (int rr = warp; rr < 2 * rank; rr += NW) {
                const __half* Am = (rr < rank ? L.Ag : L.Au) + (size_t)(rr % rank) * H + c0;
                float acc = 0.f;
                for (int c = lane * 8; c < nc; c += 256) acc += h8_dot(ldg_stream(Am + c), h + c0 + c);
                acc = warp_sum(acc);
                if (lane < TEAM) cl_st(cl_map(zred + crank * 2 * T2_MAX_RANK + rr, lane), acc);
            }
            cl_sync();
            for (int rr = tid; rr < 2 * rank; rr += T2_THREADS) {
                float v = 0.f;
                for (int m = 0; m < TEAM; ++m) v += zred[m * 2 * T2_MAX_RANK + rr];
                (rr < rank ? zg : zu)[rr % rank] = v;
            }
            __syncthreads();
        }

        // ---- gate/up rows of this member (all warps), a = silu(G h) * (U h),
        // stored into every member of the team
        {
            const RowMap rm(H, lane);
            const int step = NW * rm.R;
            for (int pb = p0 + warp * rm.R; pb < p1; pb += 2 * step) {
                uint4 c[2][4];
                uint32_t sbv[2][2];
                const uint8_t* exs[2];
                int is[2], kes[2];
                bool lv[2];
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    const int pr = pb + v * step + rm.r;
                    lv[v] = rm.active && pr < p1;
                    const int u = sp.u0 + pr / 32;
                    kes[v] = u / sp.HG;
                    is[v] = (u % sp.HG) * 32 + pr % 32;
                    exs[v] = lv[v] ? slot_s[kes[v] < K ? kes[v] : K] : nullptr;
                    if (exs[v]) {
                        const uint8_t* gp = exs[v] + (size_t)is[v] * H + 32 * rm.g;
                        c[v][0] = ldg_stream(gp);
                        c[v][1] = ldg_stream(gp + 16);
                        c[v][2] = ldg_stream(gp + H / 2);
                        c[v][3] = ldg_stream(gp + H / 2 + 16);
                        sbv[v][0] = ldg_u32(exs[v] + sl.gu_sb() + ((size_t)(2 * is[v]) * GH + rm.g) * 4);
                        sbv[v][1] = ldg_u32(exs[v] + sl.gu_sb() + ((size_t)(2 * is[v] + 1) * GH + rm.g) * 4);
                    }
                }
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    const int pr = pb + v * step + rm.r;
                    float pg = 0.f, pu = 0.f;
                    if (exs[v]) {
                        pg = q4_group_dot(c[v][0], c[v][1], hpl + rm.g, hxg[rm.g], sbv[v][0], GH);
                        pu = q4_group_dot(c[v][2], c[v][3], hpl + rm.g, hxg[rm.g], sbv[v][1], GH);
                    }
                    pg = seg_sum(pg, rm.G, lane);
                    pu = seg_sum(pu, rm.G, lane);
                    const int lead = lane - rm.g;
                    float a = 0.f;
                    if (lv[v] && rm.g == 0 && exs[v]) {
                        if (kes[v] == K && lora) {
                            float dg = 0.f, du = 0.f;
                            for (int rr = 0; rr < rank; ++rr) {
                                dg = fmaf(__half2float(L.Bg[(size_t)is[v] * rank + rr]), zg[rr], dg);
                                du = fmaf(__half2float(L.Bu[(size_t)is[v] * rank + rr]), zu[rr], du);
                            }
                            pg = fmaf(L.lscale, dg, pg);
                            pu = fmaf(L.lscale, du, pu);
                        }
                        a = silu_f(pg) * pu;
                    }
                    const float av = __shfl_sync(0xffffffffu, a, lead < 0 ? 0 : lead);
                    const int mrk = lane - lead;
                    if (lv[v] && mrk < TEAM && mrk < rm.G) cl_st(cl_map(ateam + pr, mrk), av);
                    if (lv[v] && rm.G < TEAM && rm.g == 0)
                        for (int m = rm.G; m < TEAM; ++m) cl_st(cl_map(ateam + pr, m), av);
                }
            }
        }

        // ---- the next layer's weights start moving into L2 now (this CTA's share)
        if (l + 1 < Lz) {
            const LayerP N = S.layers[l + 1];
            if (!layer_native(S, N, t)) {
                for (int k = 0; k < K; ++k) prefetch_share_lines(slot_all[(l + 1) * (K + 1) + k], sbytes, b, nb);
            } else if (N.W_r) {
                prefetch_share_lines(N.W_r, (size_t)E * H * 2, b, nb);
            }
            if (N.sh) prefetch_share_lines(N.sh, sbytes, b, nb);
            if (N.fc1) {
                prefetch_share_lines(N.fc1, (size_t)N.hidden * (H + 2 * E) * 2, b, nb);
                prefetch_share_lines(N.lres, (size_t)E * (H + 2 * E) * 2, b, nb);
            }
            if (L.fc1) prefetch_share_lines(L.fc2, (size_t)E * L.hidden * 2, b, nb);
        }

        // ---- team exchange of the activations
        cl_sync();

        // quantise the team's activations (one half-group per warp) and the
        // LoRA B input zd = A_down[:, team cols] . a_s of the shared rows
        const int nu = sp.u1 - sp.u0;
        for (int u = warp; u < nu; u += NW) quantize_half_warp(ateam[u * 32 + lane], apl + u * 4, axg + u, lane);
        if (team_lora) {
            const int us0 = max(sp.u0, K * sp.HG);
            for (int rr = warp; rr < rank; rr += NW) {
                float acc = 0.f;
                for (int p = (us0 - sp.u0) * 32 + lane; p < sp.rows; p += 32) {
                    const int i = ((sp.u0 + p / 32) % sp.HG) * 32 + p % 32;
                    acc = fmaf(__half2float(L.Ad[(size_t)rr * I + i]), ateam[p], acc);
                }
                acc = warp_sum(acc);
                if (lane == 0) zd[rr] = acc;
            }
        }
        __syncthreads();

        const int rows_m = H / TEAM;              // output rows of this member
        const int ndw = (rows_m + 31) / 32;       // warps on the down rows
        if (warp < ndw) {
            // ---- down rows: lane = output row, partial over the team's columns
            const int j = crank * rows_m + warp * 32 + lane;
            const bool live = warp * 32 + lane < rows_m;
            float acc = 0.f;
            for (int ub = sp.u0; ub < sp.u1; ub += 8) {
                uint4 cv[8];
                uint32_t sbv[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int u = ub + q;
                    const uint8_t* ex = (live && u < sp.u1) ? slot_s[u / sp.HG < K ? u / sp.HG : K] : nullptr;
                    if (ex) {
                        const int hg = u % sp.HG;
                        cv[q] = ldg_stream(ex + sl.down_codes() + ((size_t)hg * H + j) * 16);
                        sbv[q] = ldg_u32(ex + sl.down_sb() + ((size_t)(hg / 2) * H + j) * 4);
                    }
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int u = ub + q;
                    if (!live || u >= sp.u1) continue;
                    const int ke = u / sp.HG;
                    if (!slot_s[ke < K ? ke : K]) continue;
                    const float d = q4_half_dot(cv[q], apl + (u - sp.u0) * 4, axg[u - sp.u0], sbv[q]);
                    acc = fmaf(ke < K ? w_s[ke] : 1.f, d, acc);
                }
            }
            if (team_lora && live) {
                float d = 0.f;
                for (int rr = 0; rr < rank; ++rr) d = fmaf(__half2float(L.Bd[(size_t)j * rank + rr]), zd[rr], d);
                acc = fmaf(L.lscale, d, acc);
            }
            if (live && nu > 0)
                asm volatile("red.global.add.f32 [%0], %1;" ::"l"(S.y_acc + (size_t)(l % 3) * H + j), "f"(acc)
                             : "memory");
        } else {
            // ---- prerouter heads on the remaining warps: routing of owner
            // l-2's logits, fc2 of owner l-1, fc1 and the linear residual of owner l
            const int hw = NW - ndw;
            const int aw = b * hw + (warp - ndw), naw = nb * hw;
            if (b == 0 && warp == ndw && l >= 2 && S.layers[l - 2].fc1)
                stack_route_head(S, l - 2, t, scr, tr, st, lane, S.z2 + (size_t)((l - 1) & 1) * E);
            const LayerP P = l >= 1 ? S.layers[l - 1] : L;
            const int hidP = (l >= 1 && P.fc1) ? P.hidden : 0;
            const int n_fc2 = hidP > 0 ? E : 0;
            const int n_fc1 = L.fc1 ? L.hidden : 0;
            const int n_lres = L.fc1 ? E : 0;
            const int32_t* prev = t > 0 ? S.hist + ((size_t)((t + 1) & 1) * Lz + l) * K : nullptr;
            for (int it = aw; it < n_fc2 + n_fc1 + n_lres; it += naw) {
                if (it < n_fc2) {
                    const int e = it;
                    const float acc = warp_sum(
                        hrow_dot_gelu(P.fc2 + (size_t)e * hidP, S.hpre2 + (size_t)((l - 1) & 1) * hidP, hidP, lane));
                    if (lane == 0)
                        S.z2[(size_t)(l & 1) * E + e] = acc + (P.b2 ? __half2float(P.b2[e]) : 0.f) +
                                                        __ldcg(S.zres2 + (size_t)((l - 1) & 1) * E + e);
                } else {
                    const int q = it - n_fc2;
                    const bool is_fc1 = q < n_fc1;
                    const int row = is_fc1 ? q : q - n_fc1;
                    const __half* wr = (is_fc1 ? L.fc1 : L.lres) + (size_t)row * ((size_t)H + 2 * E);
                    float acc = hrow_dot(wr, h, H, lane);
                    // the one-hot columns: this layer's experts, then the previous token's
                    if (lane < 2 * K) {
                        const int e = lane < K ? inds_s[lane] : (prev ? __ldcg(prev + lane - K) : -1);
                        if (e >= 0 && e < E) acc += __half2float(wr[(lane < K ? (size_t)H : (size_t)H + E) + e]);
                    }
                    acc = warp_sum(acc);
                    if (lane == 0) {
                        if (is_fc1)
                            S.hpre2[(size_t)(l & 1) * L.hidden + row] = acc + (L.b1 ? __half2float(L.b1[row]) : 0.f);
                        else
                            S.zres2[(size_t)(l & 1) * E + row] = acc;
                    }
                }
            }
        }
        grid_barrier2(Sp, bar0 + (unsigned long long)(++nbar) * nb, st);
    }

    // ---- token output, the last pending prediction, bookkeeping
    if (b == 0) {
        const float* ysrc = S.y_acc + (size_t)((Lz - 1) % 3) * H;
        for (int j = tid; j < H; j += T2_THREADS) {
            const float v = r[j] + __ldcg(ysrc + j);
            r_out[j] = v;
            if (tr.r) tr.r[(size_t)Lz * H + j] = v;
        }
        if (warp == 1 && Lz >= 2 && S.layers[Lz - 2].fc1)
            stack_route_head(S, Lz - 2, t, scr, tr, st, lane, S.z2 + (size_t)((Lz - 1) & 1) * E);
        __syncthreads();
        // layer 0 of the next token accumulates into buffer 0
        for (int j = tid; j < H; j += T2_THREADS) S.y_acc[j] = 0.f;
        if (tid == 0) {
            S.t = t + 1;
            S.bar_base = bar0 + (unsigned long long)nbar * nb;
        }
    }
}
