// One decode token over all layers in one launch, one grid barrier per layer.
//
// The launch is made of teams: thread-block clusters of TEAM CTAs (one CTA
// per SM).  Each layer's expert work — the K routed experts plus the shared
// expert — is cut into half-groups of 32 intermediate rows; every team takes
// a contiguous run of half-groups (shared-expert units with LoRA count
// double).  Inside a team each CTA computes a slice of the SwiGLU activations
// a = silu(G h) * (U h) for the team's rows and writes them into every team
// member's shared memory (distributed shared memory); one cluster barrier
// later every member holds the team's activations, quantises them, and
// computes the partial down projection sum_k w_k D_k[:, team columns] a_k for
// its share of the output rows.  The partial sums are added into the layer
// output y with red.add; the grid barrier at the end of the layer is the only
// grid-wide synchronisation (native-routing layers add one for the router
// logits).
//
// Every CTA keeps the residual stream r in its own shared memory and
// updates it from y at the start of the next layer, so the RMSNorm needs one
// 8 KB read per CTA and no extra barrier.  The prerouter heads run on four
// head warps per CTA alongside the eight expert warps (which join once their
// down rows are done): fc2 of owner l-1 (its hidden vector is complete once
// layer l starts), fc1 and the linear residual of owner l, and the routing
// of owner l-2's logits.
//
// Each member's weight slices of a layer (gate/up row runs, down slices and
// the LoRA operands) are copied into shared memory with bulk copies: for a
// layer whose routing is a prediction made one token earlier, while the
// previous layer still runs; for a native layer, right after its routing.
// Included inside namespace e0 of e0_decode.cu (it uses StackHdr and the
// phase helpers defined there).
#pragma once

constexpr int TEAM = 8;             // CTAs per cluster
constexpr int T2_THREADS = 384;     // 12 warps
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

// ------------------------------------------------------------------ barrier

// Grid barrier on a 64-bit monotonic counter: arrive with a release add,
// wait with acquire loads until the counter reaches the target; gives up
// after a bounded number of polls (or when another CTA already did),
// raising E0_ST_TIMEOUT.  (A two-level form — cluster barrier, one arrival
// per team, cluster barrier — measured ~0.5 us slower per layer.)
E0_DEV void grid_barrier2(StackHdr* S, unsigned long long target, uint32_t* st) {
    __syncthreads();
    if (threadIdx.x == 0) {
        // the block barrier above orders every thread's writes before this
        // release, which makes them visible to whoever acquires the count
        asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(&S->bar_ctr), "l"(1ull) : "memory");
        uint32_t it = 0;
        while (true) {
            unsigned long long v;
            asm volatile("ld.acquire.gpu.u64 %0, [%1];" : "=l"(v) : "l"(&S->bar_ctr) : "memory");
            if (v >= target) break;
            if ((++it & 63u) == 0) {  // the abort flag is polled less often
                unsigned ab;
                asm volatile("ld.relaxed.gpu.u32 %0, [%1];" : "=r"(ab) : "l"(&S->bar_abort) : "memory");
                if (ab) break;
            }
            if (it > (1u << 24)) {
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
// shared-memory reads of neighbouring lanes do not collide.  Four such loads
// are in flight at a time: more would raise the kernel's register peak, and
// its spills cost more than the extra round trip.  Sum the lanes with warp_sum.
E0_DEV float hrow_dot(const __half* w, const float* x, int n, int lane) {
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

// Up to four consecutive fp16 rows (row stride ld halves) of the head's second
// layer times gelu_erf(hp), hp written by other blocks earlier in the launch
// (read from L2); the activation is evaluated once for all rows.  One chunk
// of 256 columns at a time: this is off the layer's critical path, and more
// loads in flight here set the kernel's register peak.
E0_DEV void hrow_dot_gelu4(const __half* w, size_t ld, int nrows, const float* hp, int n, int lane,
                                            float* acc) {
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c0 = 0; c0 < n; c0 += 256) {
        uint4 wv[4][1];
        float4 a[1], b[1];
#pragma unroll
        for (int k = 0; k < 1; ++k) {
            const int c = c0 + k * 256 + lane * 8;
            if (c < n) {
                a[k] = __ldcg(reinterpret_cast<const float4*>(hp + c));
                b[k] = __ldcg(reinterpret_cast<const float4*>(hp + c + 4));
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (q < nrows) wv[q][k] = ldg_stream(w + (size_t)q * ld + c);
            }
        }
#pragma unroll
        for (int k = 0; k < 1; ++k) {
            const int c = c0 + k * 256 + lane * 8;
            if (c < n) {
                const float4 ga = make_float4(gelu_erf_f(a[k].x), gelu_erf_f(a[k].y), gelu_erf_f(a[k].z), gelu_erf_f(a[k].w));
                const float4 gb = make_float4(gelu_erf_f(b[k].x), gelu_erf_f(b[k].y), gelu_erf_f(b[k].z), gelu_erf_f(b[k].w));
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (q < nrows) s[q] += h8_dot44(wv[q][k], ga, gb);
            }
        }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = s[q];
}

// ------------------------------------------------------------------ staging of weight slices

constexpr int T2_EXPERT_W = 8;   // warps 0..7: experts; 8..11: prerouter heads and staging
constexpr int T2_RES_BATCH = 4;  // residual groups a warp loads at once
constexpr size_t T2_SMEM_BUDGET = 128 * 1024;  // default shared memory of a block
constexpr int T2_SPLIT_HEAVY = 5;  // cost of a LoRA-carrying shared unit in the split (routed = 2)
// gate/up rows a warp loads before it computes: one row keeps the fewest
// values live (spills cost more here than the longer chain of rows)
constexpr int T2_GU_BATCH = 1;
constexpr int T2_MAX_SEG = 4;    // gate/up row runs of one member (one per expert touched)

constexpr int T2_STAGE_RANK = 16;   // LoRA ranks up to this are staged; larger ones read global memory
constexpr int T2_STAGE_ROUNDS = 3;  // up to 96 ranges per side and layer
constexpr int T2_STAGE_MAX = 32 * T2_STAGE_ROUNDS;

// Sources of a staged range: the slots of the K routed experts (0..K-1) and of
// the shared expert (K), then the LoRA matrices.
enum { SRC_AG = 1, SRC_AU, SRC_BG, SRC_BU, SRC_AD, SRC_BD };  // added to K

// One range of a layer's weights: `bytes` at byte offset `off` from source
// `kind`, copied to byte `soff` of the staging region (soff < 0: read in place).
struct StageEnt {
    uint64_t off;
    uint32_t bytes;
    int32_t kind;
    int32_t soff;
    int32_t pad;
};

// The ranges of one side of a layer for this member.  They depend only on the
// layer's configuration (shared expert or not, LoRA staged or not), not on
// its routing, so they are laid out once per configuration.
struct StageTab {
    int cfg;  // configuration the table was built for (-1: none yet)
    int n;
    StageEnt e[T2_STAGE_MAX];
};

// Where this CTA's weight slices of a layer are read from (a staging region of
// shared memory, or global memory), in the order of the tables.  Gate/up side
// (one region, one layer at a time): 2 * n_gu pointers for the row runs
// (codes, (scale, bias)), 2 * ra rows of LoRA A_gate then A_up (from the
// member's first column), then LoRA B_gate, B_up from the member's first
// shared row (when bsh).  Down side (two regions, by layer parity): 2 * nu
// pointers for the down slices (codes, (scale, bias)), rd rows of LoRA A_down
// (from the team's first shared column), then LoRA B_down from the member's
// first output row (when rd > 0).
struct StagePlan {
    StageTab gut, dnt;
    int n_gu, gu_pos[T2_MAX_SEG + 1], ra, bsh;  // gu_pos: first team position of each run; [n_gu] = end
    const uint8_t* gu[T2_STAGE_MAX];
    int dn_nu, dn_rd;  // of the down table
    int nu[2], rd[2];  // of the layer each down region holds
    const uint8_t* dn[2][T2_STAGE_MAX];
    E0_DEV const uint8_t* gu_codes(int n) const { return gu[2 * n]; }
    E0_DEV const uint8_t* gu_sb(int n) const { return gu[2 * n + 1]; }
    E0_DEV const __half* ag(int q) const { return ra ? reinterpret_cast<const __half*>(gu[2 * n_gu + q]) : nullptr; }
    E0_DEV const __half* bg() const { return bsh ? reinterpret_cast<const __half*>(gu[2 * n_gu + 2 * ra]) : nullptr; }
    E0_DEV const __half* bu() const { return bsh ? reinterpret_cast<const __half*>(gu[2 * n_gu + 2 * ra + 1]) : nullptr; }
    E0_DEV const uint8_t* dn_codes(int b, int u) const { return dn[b][2 * u]; }
    E0_DEV const uint8_t* dn_sb(int b, int u) const { return dn[b][2 * u + 1]; }
    E0_DEV const __half* ad(int b, int q) const {
        return rd[b] ? reinterpret_cast<const __half*>(dn[b][2 * nu[b] + q]) : nullptr;
    }
    E0_DEV const __half* bd(int b) const {
        return rd[b] ? reinterpret_cast<const __half*>(dn[b][2 * nu[b] + rd[b]]) : nullptr;
    }
};

E0_DEV void fence_async_smem2() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// weight slices are read once from HBM: evict-first in L2
E0_DEV void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            (uint32_t)__cvta_generic_to_shared(dst)),
        "l"(src), "r"(bytes), "r"((uint32_t)__cvta_generic_to_shared(bar)), "l"(l2_evict_first())
        : "memory");
}
// Bulk prefetch of a global range into L2 (16-byte aligned, size a multiple
// of 16); a hint with nothing to wait for.
E0_DEV void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
E0_DEV void mbar_init2(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"((uint32_t)__cvta_generic_to_shared(bar)), "r"(count)
                 : "memory");
}
E0_DEV void mbar_expect2(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(bar)),
                 "r"(bytes)
                 : "memory");
}
// Bounded wait for a staging barrier's phase: gives up (false) after 50 ms of
// device time; a copy of a few hundred KB lands in microseconds.
E0_DEV bool mbar_wait2(uint64_t* bar, uint32_t parity) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(bar);
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (uint32_t it = 0;; ++it) {
        if ((it & 63) == 63) {
            uint64_t t1;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
            if (t1 - t0 > 50000000ull) return false;
        }
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(a), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// Lays out the ranges of one side (item(i) gives range i as {kind, off,
// bytes}): taken in order while the running total of stageable bytes fits in
// cap; a range that is not whole 16-byte chunks at a 16-byte offset, or that
// comes after the region is full, is read in place.  One warp.
template <class Item>
E0_DEV void stage_layout(StageTab* tab, int cfg, int n, Item item, size_t cap, int lane) {
    uint32_t base = 0;
    for (int r = 0; r < T2_STAGE_ROUNDS; ++r) {
        const int i = r * 32 + lane;
        StageEnt e{0ull, 0u, -1, -1, 0};
        if (i < n) item(i, e);
        const bool ok = i < n && e.bytes > 0 && !(e.bytes & 15u) && !(e.off & 15ull);
        const uint32_t sz = ok ? e.bytes : 0u;
        uint32_t inc = sz;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        e.soff = (ok && (size_t)base + inc <= cap) ? (int32_t)(base + inc - sz) : -1;
        base += __shfl_sync(0xffffffffu, inc, 31);
        if (i < n) tab->e[i] = e;
    }
    if (lane == 0) {
        tab->n = n;
        tab->cfg = cfg;
    }
    __syncwarp();
}

// Issues one side of a layer from its table: slots[0..K] and the LoRA
// matrices are the layer's sources; rec[i] receives where range i is read from.  One warp; completes on
// `bar` with one arrival plus the bytes copied.  Every record happens before
// the arrival.
struct LoraPtrs {
    const __half *Ag, *Au, *Bg, *Bu, *Ad, *Bd;
};

E0_DEV void stage_issue(const StageTab* tab, const uint8_t* const* slots, int K, const LoraPtrs& lo, uint8_t* buf,
                        const uint8_t** rec, uint64_t* bar, int lane) {
    const uint8_t* from[T2_STAGE_ROUNDS];
    int32_t to[T2_STAGE_ROUNDS];
    uint32_t nbytes[T2_STAGE_ROUNDS];
    uint32_t tot = 0;
    const int n = tab->n;
#pragma unroll
    for (int r = 0; r < T2_STAGE_ROUNDS; ++r) {
        const int i = r * 32 + lane;
        from[r] = nullptr;
        to[r] = -1;
        nbytes[r] = 0;
        if (i < n) {
            const StageEnt e = tab->e[i];
            const void* bv = nullptr;
            switch (e.kind - K) {
                case SRC_AG: bv = lo.Ag; break;
                case SRC_AU: bv = lo.Au; break;
                case SRC_BG: bv = lo.Bg; break;
                case SRC_BU: bv = lo.Bu; break;
                case SRC_AD: bv = lo.Ad; break;
                case SRC_BD: bv = lo.Bd; break;
                default: bv = slots[e.kind];
            }
            const uint8_t* b = reinterpret_cast<const uint8_t*>(bv);
            const uint8_t* p = b ? b + e.off : nullptr;
            const bool al = p && !(reinterpret_cast<uintptr_t>(p) & 15u);
            const bool cp = al && e.soff >= 0;
            rec[i] = cp ? buf + e.soff : p;
            // a range left in global memory is brought into L2 now, so that its
            // reads later in the layer hit L2 instead of HBM
            if (al && !cp && e.bytes > 0 && !(e.bytes & 15u)) prefetch_l2(p, e.bytes);
            if (cp) {
                from[r] = p;
                to[r] = e.soff;
                nbytes[r] = e.bytes;
                tot += e.bytes;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    // the region's previous contents were read by the generic proxy
    fence_async_smem2();
    __syncwarp();
    if (lane == 0) mbar_expect2(bar, tot);
    __syncwarp();
#pragma unroll
    for (int r = 0; r < T2_STAGE_ROUNDS; ++r)
        if (to[r] >= 0) bulk_copy(buf + to[r], from[r], nbytes[r], bar);
}

// Gate/up side: the row runs of team positions [p0, p1) (one run per expert
// touched; consecutive positions of one expert are consecutive rows of its
// slot: codes, then (scale, bias) words), the member's column slice
// [c0, c0 + nc) of the ra rows of LoRA A_gate and A_up, and the LoRA B_gate /
// B_up rows of its shared-expert positions [ps, p1) (first row i_s).
__device__ __noinline__ void stage_layout_gu(StagePlan* plan, int cfg, const SlotLayout& sl, int H, int K, int HG,
                                             int u0, int p0, int p1, int ra, int rank, int c0, int nc, int ps, int i_s,
                                             size_t cap, int lane) {
    const int GH = H / GROUP;
    const int ke0 = (u0 + p0 / 32) / HG;
    const int nrun = p1 > p0 ? (u0 + (p1 - 1) / 32) / HG - ke0 + 1 : 0;
    const int n_gu = nrun < T2_MAX_SEG ? nrun : T2_MAX_SEG;
    const bool bsh = ra > 0 && ps < p1;
    auto run_start = [&](int n) { return max(p0, ((ke0 + n) * HG - u0) * 32); };
    auto run_end = [&](int n) { return min(p1, ((ke0 + n + 1) * HG - u0) * 32); };
    auto item = [&](int i, StageEnt& e) {
        if (i < 2 * n_gu) {
            const int n = i >> 1;
            const int pst = run_start(n), rows = run_end(n) - pst;
            const int ia = ((u0 + pst / 32) % HG) * 32 + pst % 32;
            e.kind = min(ke0 + n, K);
            if (i & 1) {
                e.off = sl.gu_sb() + (uint64_t)ia * 2 * GH * 4;
                e.bytes = (uint32_t)rows * 2 * GH * 4;
            } else {
                e.off = (uint64_t)ia * H;
                e.bytes = (uint32_t)rows * H;
            }
            return;
        }
        const int q = i - 2 * n_gu;
        if (q < 2 * ra) {
            e.kind = K + (q < ra ? SRC_AG : SRC_AU);
            e.off = ((uint64_t)(q % ra) * H + c0) * 2;
            e.bytes = (uint32_t)nc * 2;
            return;
        }
        e.kind = K + (q == 2 * ra ? SRC_BG : SRC_BU);
        e.off = (uint64_t)i_s * rank * 2;
        e.bytes = (uint32_t)(p1 - ps) * rank * 2;
    };
    if (lane == 0) {
        plan->n_gu = n_gu;
        for (int n = 0; n < n_gu; ++n) plan->gu_pos[n] = run_start(n);
        plan->gu_pos[n_gu] = n_gu > 0 ? run_end(n_gu - 1) : p0;
        plan->ra = ra;
        plan->bsh = bsh ? 1 : 0;
    }
    stage_layout(&plan->gut, cfg, 2 * n_gu + 2 * ra + (bsh ? 2 : 0), item, cap, lane);
}

// Down side: the down slices (output rows [j0, j1)) of half-group units
// [u0, u1), the team's shared columns [i0, i0 + ni) of the rd rows of LoRA
// A_down, and the member's rows of LoRA B_down.
__device__ __noinline__ void stage_layout_dn(StagePlan* plan, int cfg, const SlotLayout& sl, int H, int K, int HG,
                                             int u0, int u1, int j0, int j1, int rd, int rank, int i0, int ni,
                                             size_t cap, int lane) {
    const int nu = u1 - u0;
    auto item = [&](int i, StageEnt& e) {
        if (i < 2 * nu) {
            const int u = u0 + (i >> 1), hg = u % HG;
            e.kind = min(u / HG, K);
            if (i & 1) {
                e.off = sl.down_sb() + ((uint64_t)(hg / 2) * H + j0) * 4;
                e.bytes = (uint32_t)(j1 - j0) * 4;
            } else {
                e.off = sl.down_codes() + ((uint64_t)hg * H + j0) * 16;
                e.bytes = (uint32_t)(j1 - j0) * 16;
            }
            return;
        }
        const int q = i - 2 * nu;
        if (q < rd) {
            e.kind = K + SRC_AD;
            e.off = ((uint64_t)q * (HG * 32) + i0) * 2;
            e.bytes = (uint32_t)ni * 2;
            return;
        }
        e.kind = K + SRC_BD;
        e.off = (uint64_t)j0 * rank * 2;
        e.bytes = (uint32_t)(j1 - j0) * rank * 2;
    };
    if (lane == 0) {
        plan->dn_nu = nu;
        plan->dn_rd = rd;
    }
    stage_layout(&plan->dnt, cfg, 2 * nu + (rd > 0 ? rd + 1 : 0), item, cap, lane);
}

// Bytes one member may stage for one layer when NT teams share nk experts:
// gate/up rows (codes + scale/bias) and down slices.
__host__ __device__ inline void stage_need(int H, int I, int units, int rank, size_t* gu, size_t* dn) {
    const int rows = (units * 32 + TEAM - 1) / TEAM;
    const int r = rank <= T2_STAGE_RANK ? rank : 0;
    *gu = (size_t)rows * (H + 2 * (H / GROUP) * 4) + (size_t)T2_MAX_SEG * 64  // row runs
          + (size_t)2 * r * (H / TEAM) * 2 + (size_t)2 * rows * r * 2;       // LoRA A slices, B rows
    *dn = (size_t)units * (H / TEAM) * 20                                     // down slices
          + (size_t)r * units * 32 * 2 + (size_t)(H / TEAM) * r * 2;          // LoRA A_down, B_down
}

// ------------------------------------------------------------------ shared memory layout

struct T2Smem {
    uint32_t hdr, lyr, r, hpl, hxg, ateam, apl, axg, zred, zg, zu, zd, inds, w, slots, scr, red, hnext, plan, bars, stage_gu,
        stage_dn, dn_bytes, total;
    __host__ __device__ T2Smem(int H, int E, int L, int K, size_t gu_cap, size_t dn_cap) {
        const int GH = H / GROUP;
        const int max_rows = T2_MAX_UNITS * 32;
        size_t o = 0;
        hdr = o;  // copy of the stack header (read-only during a launch)
        o += (sizeof(StackHdr) + 15) & ~(size_t)15;
        lyr = o;  // copy of the layer descriptors
        o += ((size_t)L * sizeof(LayerP) + 15) & ~(size_t)15;
        r = o;
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
        hnext = o;  // next prerouter-head unit of this block
        o += 16;
        o = (o + 15) & ~(size_t)15;
        plan = o;
        o += sizeof(StagePlan);
        o = (o + 15) & ~(size_t)15;
        bars = o;  // [0] gate/up region, [1], [2] down regions
        o += 3 * 8;
        o = (o + 127) & ~(size_t)127;
        stage_gu = o;
        o += gu_cap;
        o = (o + 127) & ~(size_t)127;
        stage_dn = o;  // two regions of dn_cap bytes, by layer parity
        dn_bytes = dn_cap;
        o += 2 * dn_cap;
        total = (o + 127) & ~(size_t)127;
    }
};

// Work split of one layer: NU half-group units (the nk_r routed experts
// first, then the shared expert when there is one), cut into NT contiguous
// runs of about equal cost; team tau takes units [u0, u1).  A unit of a shared
// expert with LoRA costs 2.5 times a routed one by default (its team also
// computes the LoRA A and B products and waits for one more team exchange;
// 2.5 measured faster than 2 or 3 on GB300), so such teams get fewer units.
struct T2Split {
    int HG, NU, u0, u1, rows;
    // wh: cost of a shared-expert unit that carries LoRA, in halves of a
    // routed unit's cost
    __host__ __device__ static int bound(int HG, int KH, int NU, bool heavy, int wh, int tau, int NT) {
        if (!heavy) return (int)((long)tau * NU / NT);
        const long Wt = 2L * KH + (long)wh * (NU - KH);  // cost in half units
        const long w = (long)tau * Wt / NT;
        return w <= 2L * KH ? (int)(w / 2) : KH + (int)((w - 2L * KH) / wh);
    }
    // nk_r routed experts; sh: a shared expert follows; heavy: it carries LoRA
    __host__ __device__ T2Split(int I, int nk_r, bool sh, bool heavy, int wh, int tau, int NT) {
        HG = I / 32;
        const int KH = nk_r * HG;
        NU = KH + (sh ? HG : 0);
        u0 = bound(HG, KH, NU, sh && heavy, wh, tau, NT);
        u1 = bound(HG, KH, NU, sh && heavy, wh, tau + 1, NT);
        rows = (u1 - u0) * 32;
    }
};

// ------------------------------------------------------------------ the kernel

__global__ void __launch_bounds__(T2_THREADS, 1)
    k_stack_token2(StackHdr* Sp, const float* x, float* r_out, TraceP tr, uint32_t* st, int lb, int le) {
    extern __shared__ __align__(16) char smem[];
    const int H = Sp->H, I = Sp->I, E = Sp->E, K = Sp->K, Lz = Sp->L;
    const int GH = H / GROUP;
    const int t = Sp->t;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NW = T2_THREADS >> 5;
    const int nb = gridDim.x, b = blockIdx.x;
    const int team = (int)cl_id(), NT = (int)cl_count(), crank = (int)cl_rank();
    const unsigned long long bar0 = Sp->bar_base;
    int nbar = 0;

    const T2Smem lay(H, E, Lz, K, (size_t)Sp->smem2_gu, (size_t)Sp->smem2_dn);
    // The header and the layer descriptors do not change during a launch:
    // read them from shared memory.  Sp stays the place for the barrier
    // counters and the end-of-token bookkeeping.
    {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(Sp);
        uint32_t* dst = reinterpret_cast<uint32_t*>(smem + lay.hdr);
        for (int i = threadIdx.x; i < (int)(sizeof(StackHdr) / 4); i += T2_THREADS) dst[i] = src[i];
        const uint32_t* ls = reinterpret_cast<const uint32_t*>(Sp->layers);
        uint32_t* ld = reinterpret_cast<uint32_t*>(smem + lay.lyr);
        for (int i = threadIdx.x; i < (int)((size_t)Lz * sizeof(LayerP) / 4); i += T2_THREADS) ld[i] = ls[i];
        __syncthreads();
    }
    const StackHdr& S = *reinterpret_cast<const StackHdr*>(smem + lay.hdr);
    const LayerP* lyr = reinterpret_cast<const LayerP*>(smem + lay.lyr);
    float* r = reinterpret_cast<float*>(smem + lay.r);
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
    int* hnext = reinterpret_cast<int*>(smem + lay.hnext);
    StagePlan& plan = *reinterpret_cast<StagePlan*>(smem + lay.plan);
    uint64_t* sbar = reinterpret_cast<uint64_t*>(smem + lay.bars);
    uint8_t* stage_gu_buf = reinterpret_cast<uint8_t*>(smem + lay.stage_gu);
    uint8_t* stage_dn_buf = reinterpret_cast<uint8_t*>(smem + lay.stage_dn);

    const SlotLayout sl{H, I};
    const size_t sbytes = sl.bytes();
    const int rows_m = H / TEAM;  // output rows of this member
    const int j0 = crank * rows_m, j1 = j0 + rows_m;

    if (tid == 0) {
        mbar_init2(&sbar[0], 1);
        mbar_init2(&sbar[1], 1);
        mbar_init2(&sbar[2], 1);
        plan.gut.cfg = -1;
        plan.dnt.cfg = -1;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // ---- routing of every layer that takes a prediction this token (known now)
    for (int q = tid; q < Lz * (K + 1); q += T2_THREADS) {
        const int l = q / (K + 1), k = q % (K + 1);
        const LayerP& L = lyr[l];
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

    auto split_of = [&](int l) {
        const LayerP& Lq = lyr[l];
        return T2Split(I, K, Lq.sh != nullptr, Lq.sh != nullptr && Lq.Ag != nullptr, S.split_heavy, team, NT);
    };
    // Staging.  The gate/up region holds one layer at a time and completes once
    // per layer (layer l waits on parity (l - lb) & 1, counting from the first
    // layer of this launch); the down regions alternate by layer parity (layer
    // l waits on region l & 1, parity ((l - lb) >> 1) & 1).  A
    // layer whose routing is known when the token starts is copied while the
    // layer before it runs: its down side when that layer starts, its gate/up
    // side once that layer's gate/up rows have been read.  A native layer is
    // copied right after its routing.  The first head warp issues every copy.
    constexpr int HW = T2_EXPERT_W;
    // configuration key of a layer's tables: no shared expert; shared expert
    // with LoRA read in place; shared expert with LoRA of rank r staged
    auto cfg_of = [&](int l) {
        const LayerP& Lq = lyr[l];
        if (!Lq.sh) return 0;
        return (Lq.Ag && Lq.rank <= T2_STAGE_RANK) ? 2 + Lq.rank : 1;
    };
    auto lora_ptrs = [&](int l) {
        const LayerP& Lq = lyr[l];
        return LoraPtrs{Lq.Ag, Lq.Au, Lq.Bg, Lq.Bu, Lq.Ad, Lq.Bd};
    };
    auto stage_gu_for = [&](int l) {
        const int cfg = cfg_of(l);
        if (plan.gut.cfg != cfg) {
            const T2Split sp = split_of(l);
            const int p0 = (int)((long)crank * sp.rows / TEAM), p1 = (int)((long)(crank + 1) * sp.rows / TEAM);
            const int ps = max(p0, (K * sp.HG - sp.u0) * 32);
            const int i_s = ps < p1 ? ((sp.u0 + ps / 32) % sp.HG) * 32 + ps % 32 : 0;
            const int ra = (cfg >= 2 && sp.u1 > K * sp.HG) ? cfg - 2 : 0;
            stage_layout_gu(&plan, cfg, sl, H, K, sp.HG, sp.u0, p0, p1, ra, cfg - 2, crank * (H / TEAM), H / TEAM, ps,
                            i_s, lay.stage_dn - lay.stage_gu, lane);
        }
        stage_issue(&plan.gut, slot_all + l * (K + 1), K, lora_ptrs(l), stage_gu_buf, plan.gu, &sbar[0], lane);
    };
    auto stage_dn_for = [&](int l) {
        const int cfg = cfg_of(l);
        if (plan.dnt.cfg != cfg) {
            const T2Split sp = split_of(l);
            const int us0 = max(sp.u0, K * sp.HG);
            const int ni = sp.u1 > us0 ? (sp.u1 - us0) * 32 : 0;
            const int rd = (cfg >= 2 && ni > 0) ? cfg - 2 : 0;
            stage_layout_dn(&plan, cfg, sl, H, K, sp.HG, sp.u0, sp.u1, j0, j1, rd, cfg - 2, (us0 - K * sp.HG) * 32, ni,
                            lay.dn_bytes, lane);
        }
        const int b = l & 1;
        if (lane == 0) {
            plan.nu[b] = plan.dn_nu;
            plan.rd[b] = plan.dn_rd;
        }
        stage_issue(&plan.dnt, slot_all + l * (K + 1), K, lora_ptrs(l), stage_dn_buf + (size_t)b * lay.dn_bytes,
                    plan.dn[b], &sbar[1 + b], lane);
    };
    if (warp == HW && !layer_native(S, lyr[lb], t)) {
        stage_gu_for(lb);
        stage_dn_for(lb);
    }
    // a launch that starts inside the token picks up the residual stream the
    // previous launch of this token left in the header
    if (lb > 0) {
        for (int j = tid; j < H; j += T2_THREADS) r[j] = __ldcg(S.r + j);
        __syncthreads();
    }

    for (int l = lb; l < le; ++l) {
        const LayerP& L = lyr[l];
        const bool native = layer_native(S, L, t);
        const bool sh = L.sh != nullptr;
        const bool lora = sh && L.Ag != nullptr;
        const int rank = lora ? L.rank : 0;
        int32_t* inds_s = inds_all + l * K;
        float* w_s = w_all + l * K;
        const uint8_t** slot_s = slot_all + l * (K + 1);

        // ---- residual stream r_l = x (l = 0) or r_{l-1} + y_{l-1}, and the planes
        // of h = RMSNorm(r) = r / denom.  The int16 codes of a group do not
        // change when the group is scaled, so each warp quantises its groups of
        // r while it updates them, and every product with h is taken with r and
        // scaled by inv_denom afterwards (planes, router, LoRA A, head rows):
        // one pass and one block barrier.
        float inv_denom;
        {
            const float* ysrc = l == 0 ? x : S.y_acc + (size_t)((l - 1) % 3) * H;
            float ss = 0.f;
            // a warp's groups (up to T2_RES_BATCH at a time) are loaded together,
            // so their L2 reads overlap, then updated and quantised
            for (int g0 = warp; g0 < GH; g0 += T2_RES_BATCH * NW) {
                float2 v[T2_RES_BATCH];
#pragma unroll
                for (int q = 0; q < T2_RES_BATCH; ++q) {
                    const int g = g0 + q * NW;
                    if (g < GH) v[q] = __ldcg(reinterpret_cast<const float2*>(ysrc + GROUP * g + 2 * lane));
                }
#pragma unroll
                for (int q = 0; q < T2_RES_BATCH; ++q) {
                    const int g = g0 + q * NW;
                    if (g < GH) {
                        const int j = GROUP * g + 2 * lane;
                        if (l > 0) {
                            const float2 r2 = *reinterpret_cast<const float2*>(r + j);
                            v[q] = make_float2(r2.x + v[q].x, r2.y + v[q].y);
                        }
                        *reinterpret_cast<float2*>(r + j) = v[q];
                        ss = fmaf(v[q].x, v[q].x, fmaf(v[q].y, v[q].y, ss));
                        // word k of group g sits at hpl[k * GH + g]: lanes that read
                        // consecutive groups touch consecutive 16-byte words
                        quantize_group_v(v[q], hpl + g, hxg + g, lane, nullptr, GH);
                    }
                }
            }
            ss = warp_sum(ss);
            if (lane == 0) red[warp] = ss;
            // this block's prerouter-head units of layer l start from the first
            if (tid == 0) *hnext = 0;
            // the output buffer of layer l+1 starts at zero
            if (b == nb - 1)
                for (int j = tid; j < H; j += T2_THREADS) S.y_acc[(size_t)((l + 1) % 3) * H + j] = 0.f;
            __syncthreads();
            float tot = lane < NW ? red[lane] : 0.f;
            tot = warp_sum(tot);
            inv_denom = 1.f / sqrtf(tot / (float)H + 1e-6f);
            if (b == 0 && tr.r)
                for (int j = tid; j < H; j += T2_THREADS) tr.r[(size_t)l * H + j] = r[j];
        }

        // ---- routing of native layers: logits on every warp of the grid, one grid barrier
        if (native) {
            for (int e = b * NW + warp; e < E; e += nb * NW) {
                const float acc = warp_sum(hrow_dot(L.W_r + (size_t)e * H, r, H, lane));
                if (lane == 0) S.logits[e] = acc * inv_denom;
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
            if (warp == HW) {
                stage_gu_for(l);
                stage_dn_for(l);
            }
        }
        if (b == 0 && warp == 1 && lane < K) {
            const int e = inds_s[lane];
            if (!slot_s[lane]) set_status(st, (e < 0 || e >= E) ? E0_ST_BAD_EXPERT : E0_ST_SLOT_MISS);
            S.hist[((size_t)(t & 1) * Lz + l) * K + lane] = e;
            S.wcur[(size_t)l * K + lane] = w_s[lane];
            if (tr.inds) tr.inds[(size_t)l * K + lane] = e;
            if (tr.w) tr.w[(size_t)l * K + lane] = w_s[lane];
        }

        const T2Split sp = split_of(l);
        const int p0 = (int)((long)crank * sp.rows / TEAM), p1 = (int)((long)(crank + 1) * sp.rows / TEAM);
        const bool team_lora = lora && sp.u1 > K * sp.HG;
        // the next layer's slices are copied ahead only when it runs in this
        // launch: every bulk copy is waited for before the CTA exits
        const bool next_known = l + 1 < le && !layer_native(S, lyr[l + 1], t);
        const int ps_m = max(p0, (K * sp.HG - sp.u0) * 32);  // this member's first shared-expert position
        const int db = l & 1;  // down region of this layer

        // ---- LoRA A of the shared expert (teams holding shared rows): each
        // member reduces 1/TEAM of the inputs, partial sums exchanged
        if (team_lora) {
            const int c0 = crank * (H / TEAM), nc = H / TEAM;
            if (!mbar_wait2(&sbar[0], (l - lb) & 1)) set_status(st, E0_ST_TIMEOUT);
            for (int rr = warp; rr < 2 * rank; rr += NW) {
                const __half* Am =
                    plan.ag(0) ? plan.ag(rr) : (rr < rank ? L.Ag : L.Au) + (size_t)(rr % rank) * H + c0;
                float acc = 0.f;
                // Am may point into a staging region: a generic load serves either space
                for (int c = lane * 8; c < nc; c += 256)
                    acc += h8_dot(*reinterpret_cast<const uint4*>(Am + c), r + c0 + c);
                acc = warp_sum(acc);
                if (lane < TEAM) cl_st(cl_map(zred + crank * 2 * T2_MAX_RANK + rr, lane), acc);
            }
            cl_sync();
            for (int rr = tid; rr < 2 * rank; rr += T2_THREADS) {
                float v = 0.f;
                for (int m = 0; m < TEAM; ++m) v += zred[m * 2 * T2_MAX_RANK + rr];
                (rr < rank ? zg : zu)[rr % rank] = v * inv_denom;
            }
            __syncthreads();
        }

        if (warp < T2_EXPERT_W) {
            if (!mbar_wait2(&sbar[0], (l - lb) & 1)) set_status(st, E0_ST_TIMEOUT);
            // ---- gate/up rows of this member, a = silu(G h) * (U h), stored into every member
            const RowMap rm(H, lane);
            const int step = T2_EXPERT_W * rm.R;
            for (int pb = p0 + warp * rm.R; pb < p1; pb += T2_GU_BATCH * step) {
                uint4 c[T2_GU_BATCH][4];
                uint32_t sbv[T2_GU_BATCH][2];
                bool lv[T2_GU_BATCH], hv[T2_GU_BATCH];
                int is[T2_GU_BATCH], kes[T2_GU_BATCH];
#pragma unroll
                for (int v = 0; v < T2_GU_BATCH; ++v) {
                    const int pr = pb + v * step + rm.r;
                    lv[v] = rm.active && pr < p1;
                    const int u = sp.u0 + pr / 32;
                    kes[v] = u / sp.HG;
                    is[v] = (u % sp.HG) * 32 + pr % 32;
                    hv[v] = false;
                    if (lv[v]) {
                        int sg = 0;
                        while (sg < plan.n_gu && plan.gu_pos[sg + 1] <= pr) ++sg;
                        const uint8_t* cb;
                        const uint8_t* sbb;
                        int rr;
                        if (sg < plan.n_gu) {
                            cb = plan.gu_codes(sg);
                            sbb = plan.gu_sb(sg);
                            rr = pr - plan.gu_pos[sg];
                        } else {  // beyond the staged runs: the slot in global memory
                            const uint8_t* ex = slot_s[kes[v] < K ? kes[v] : K];
                            cb = ex;
                            sbb = ex ? ex + sl.gu_sb() : nullptr;
                            rr = is[v];
                        }
                        if (cb && sbb) {
                            const uint8_t* gp = cb + (size_t)rr * H + 32 * rm.g;
                            c[v][0] = *reinterpret_cast<const uint4*>(gp);
                            c[v][1] = *reinterpret_cast<const uint4*>(gp + 16);
                            c[v][2] = *reinterpret_cast<const uint4*>(gp + H / 2);
                            c[v][3] = *reinterpret_cast<const uint4*>(gp + H / 2 + 16);
                            const uint8_t* sp2 = sbb + (size_t)rr * 2 * GH * 4 + rm.g * 4;
                            sbv[v][0] = *reinterpret_cast<const uint32_t*>(sp2);
                            sbv[v][1] = *reinterpret_cast<const uint32_t*>(sp2 + GH * 4);
                            hv[v] = true;
                        }
                    }
                }
#pragma unroll
                for (int v = 0; v < T2_GU_BATCH; ++v) {
                    const int pr = pb + v * step + rm.r;
                    float pg = 0.f, pu = 0.f;
                    if (hv[v]) {
                        pg = q4_group_dot(c[v][0], c[v][1], hpl + rm.g, hxg[rm.g], sbv[v][0], GH);
                        pu = q4_group_dot(c[v][2], c[v][3], hpl + rm.g, hxg[rm.g], sbv[v][1], GH);
                    }
                    pg = seg_sum(pg, rm.G, lane) * inv_denom;
                    pu = seg_sum(pu, rm.G, lane) * inv_denom;
                    const int lead = lane - rm.g;
                    float a = 0.f;
                    if (lv[v] && rm.g == 0 && hv[v]) {
                        if (kes[v] == K && lora) {
                            float dg = 0.f, du = 0.f;
                            const __half* bgr = plan.bg() ? plan.bg() + (size_t)(pr - ps_m) * rank : L.Bg + (size_t)is[v] * rank;
                            const __half* bur = plan.bu() ? plan.bu() + (size_t)(pr - ps_m) * rank : L.Bu + (size_t)is[v] * rank;
                            for (int rr = 0; rr < rank; ++rr) {
                                dg = fmaf(__half2float(bgr[rr]), zg[rr], dg);
                                du = fmaf(__half2float(bur[rr]), zu[rr], du);
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
            // this CTA's gate/up side has been read: the issuing head warp may
            // bring in the next layer's
            asm volatile("bar.arrive 2, %0;" ::"r"(T2_EXPERT_W * 32 + 32));
            // ---- team exchange of the activations
            cl_sync();
            if (!mbar_wait2(&sbar[1 + (l & 1)], ((l - lb) >> 1) & 1)) set_status(st, E0_ST_TIMEOUT);
            // quantise the team's activations (one half-group per warp) and the
            // LoRA B input zd = A_down[:, team cols] . a_s of the shared rows
            const int nu = sp.u1 - sp.u0;
            for (int u = warp; u < nu; u += T2_EXPERT_W) quantize_half_warp(ateam[u * 32 + lane], apl + u * 4, axg + u, lane);
            if (team_lora) {
                const int us0 = max(sp.u0, K * sp.HG);
                for (int rr = warp; rr < rank; rr += T2_EXPERT_W) {
                    float acc = 0.f;
                    const int i0t = (us0 - K * sp.HG) * 32;  // the team's first shared column
                    for (int p = (us0 - sp.u0) * 32 + lane; p < sp.rows; p += 32) {
                        const int i = ((sp.u0 + p / 32) % sp.HG) * 32 + p % 32;
                        const float ad = plan.ad(db, 0) ? __half2float(plan.ad(db, rr)[i - i0t])
                                                        : __half2float(L.Ad[(size_t)rr * I + i]);
                        acc = fmaf(ad, ateam[p], acc);
                    }
                    acc = warp_sum(acc);
                    if (lane == 0) zd[rr] = acc;
                }
            }
            asm volatile("bar.sync 1, %0;" ::"r"(T2_EXPERT_W * 32));
            // ---- down rows: lane = output row, partial over the team's columns
            // (four half-group units in flight: the register peak, as above)
            for (int jr = warp * 32 + lane; jr - lane < rows_m; jr += T2_EXPERT_W * 32) {
                if (jr >= rows_m) continue;
                const int j = j0 + jr;
                float acc = 0.f;
                for (int ub = sp.u0; ub < sp.u1; ub += 4) {
                    uint4 cv[4];
                    uint32_t sbv[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int u = ub + q;
                        if (u < sp.u1 && plan.dn_codes(db, u - sp.u0) && plan.dn_sb(db, u - sp.u0)) {
                            cv[q] = *reinterpret_cast<const uint4*>(plan.dn_codes(db, u - sp.u0) + (size_t)jr * 16);
                            sbv[q] = *reinterpret_cast<const uint32_t*>(plan.dn_sb(db, u - sp.u0) + (size_t)jr * 4);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int u = ub + q;
                        if (u >= sp.u1 || !plan.dn_codes(db, u - sp.u0) || !plan.dn_sb(db, u - sp.u0)) continue;
                        const int ke = u / sp.HG;
                        const float d = q4_half_dot(cv[q], apl + (u - sp.u0) * 4, axg[u - sp.u0], sbv[q]);
                        acc = fmaf(ke < K ? w_s[ke] : 1.f, d, acc);
                    }
                }
                if (team_lora) {
                    float d = 0.f;
                    const __half* bdr = plan.bd(db) ? plan.bd(db) + (size_t)jr * rank : L.Bd + (size_t)j * rank;
                    for (int rr = 0; rr < rank; ++rr) d = fmaf(__half2float(bdr[rr]), zd[rr], d);
                    acc = fmaf(L.lscale, d, acc);
                }
                if (nu > 0)
                    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(S.y_acc + (size_t)(l % 3) * H + j), "f"(acc)
                                 : "memory");
            }
        } else {
            // ---- head warps: nothing they do feeds the team exchange, so they
            // arrive at it now and wait at the end of the layer
            cl_arrive();
            // the next layer's down side goes to the other down region now
            if (warp == HW && next_known) stage_dn_for(l + 1);
            // a next layer that routes natively: the router rows this block will
            // compute are brought into L2 now
            if (warp == HW + 2 && lane == 0 && l + 1 < le && layer_native(S, lyr[l + 1], t)) {
                const int e0 = b * NW, ne = min(NW, E - e0);
                const __half* wr = lyr[l + 1].W_r + (size_t)e0 * H;
                if (ne > 0 && !(reinterpret_cast<uintptr_t>(wr) & 15u) && !((H * 2) & 15))
                    prefetch_l2(wr, (uint32_t)ne * H * 2);
            }
            // one warp of the last block (not the issuing one) routes owner l-2's logits
            if (b == nb - 1 && warp == HW + 1 && l >= 2 && lyr[l - 2].fc1)
                stack_route_head(S, l - 2, t, scr, tr, st, lane, S.z2 + (size_t)((l - 1) & 1) * E);
        }

        // ---- prerouter heads: fc2 of owner l-1 (four rows a unit) and fc1 /
        // linear residual of owner l (one row a unit).  This block's units are
        // handed out one at a time: the head warps start right away, the expert
        // warps join once their down rows are done.
        {
            const LayerP& P = l >= 1 ? lyr[l - 1] : L;
            const int hidP = (l >= 1 && P.fc1) ? P.hidden : 0;
            const int n_fc2 = hidP > 0 ? E : 0;
            const int n_fc1 = L.fc1 ? L.hidden : 0;
            const int n_row = L.fc1 ? L.hidden + E : 0;  // fc1 rows, then linear-residual rows
            const int nA = (n_fc2 + 3) / 4;
            const int n_units = nA + n_row;
            const int32_t* prev = t > 0 ? S.hist + ((size_t)((t + 1) & 1) * Lz + l) * K : nullptr;
            while (true) {
                // this block takes units b, b + nb, b + 2 nb, ...: the four-row
                // fc2 units (first in the numbering) spread over all blocks
                int it = 0;
                if (lane == 0) it = b + nb * atomicAdd(hnext, 1);
                it = __shfl_sync(0xffffffffu, it, 0);
                if (it >= n_units) break;
                if (it < nA) {
                    const int e0 = 4 * it, nr = min(4, n_fc2 - e0);
                    float acc[4];
                    hrow_dot_gelu4(P.fc2 + (size_t)e0 * hidP, (size_t)hidP, nr, S.hpre2 + (size_t)((l - 1) & 1) * hidP,
                                   hidP, lane, acc);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float v = warp_sum(acc[q]);
                        if (lane == 0 && q < nr)
                            S.z2[(size_t)(l & 1) * E + e0 + q] = v + (P.b2 ? __half2float(P.b2[e0 + q]) : 0.f) +
                                                                 __ldcg(S.zres2 + (size_t)((l - 1) & 1) * E + e0 + q);
                    }
                } else {
                    const int q = it - nA;
                    const __half* wr = q < n_fc1 ? L.fc1 + (size_t)q * ((size_t)H + 2 * E)
                                                 : L.lres + (size_t)(q - n_fc1) * ((size_t)H + 2 * E);
                    float a0 = hrow_dot(wr, r, H, lane) * inv_denom;
                    // the one-hot columns: this layer's experts, then the previous token's
                    if (lane < 2 * K) {
                        const int e = lane < K ? inds_s[lane] : (prev ? __ldcg(prev + lane - K) : -1);
                        if (e >= 0 && e < E) a0 += __half2float(wr[(lane < K ? (size_t)H : (size_t)H + E) + e]);
                    }
                    a0 = warp_sum(a0);
                    if (lane == 0) {
                        if (q < n_fc1)
                            S.hpre2[(size_t)(l & 1) * L.hidden + q] = a0 + (L.b1 ? __half2float(L.b1[q]) : 0.f);
                        else
                            S.zres2[(size_t)(l & 1) * E + (q - n_fc1)] = a0;
                    }
                }
            }
        }
        if (warp >= T2_EXPERT_W) {
            if (warp == HW) {
                // wait until this CTA's gate/up side has been read, then bring in the next layer's
                asm volatile("bar.sync 2, %0;" ::"r"(T2_EXPERT_W * 32 + 32));
                if (next_known) stage_gu_for(l + 1);
            }
            cl_wait();
        }
        grid_barrier2(Sp, bar0 + (unsigned long long)(++nbar) * nb, st);
    }

    if (le < Lz) {
        // ---- the token continues in another launch: hand over r_{le-1}
        if (b == 0) {
            for (int j = tid; j < H; j += T2_THREADS) S.r[j] = r[j];
            if (tid == 0) Sp->bar_base = bar0 + (unsigned long long)nbar * nb;
        }
        return;
    }
    // ---- token output, the last pending prediction, bookkeeping
    if (b == 0) {
        const float* ysrc = S.y_acc + (size_t)((Lz - 1) % 3) * H;
        for (int j = tid; j < H; j += T2_THREADS) {
            const float v = r[j] + __ldcg(ysrc + j);
            r_out[j] = v;
            if (tr.r) tr.r[(size_t)Lz * H + j] = v;
        }
        if (warp == 1 && Lz >= 2 && lyr[Lz - 2].fc1)
            stack_route_head(S, Lz - 2, t, scr, tr, st, lane, S.z2 + (size_t)((Lz - 1) & 1) * E);
        __syncthreads();
        // layer 0 of the next token accumulates into buffer 0
        for (int j = tid; j < H; j += T2_THREADS) S.y_acc[j] = 0.f;
        if (tid == 0) {
            Sp->t = t + 1;
            Sp->bar_base = bar0 + (unsigned long long)nbar * nb;
        }
    }
}
