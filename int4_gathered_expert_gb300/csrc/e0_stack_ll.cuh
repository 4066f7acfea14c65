// One decode token over layers [lb, le) in one cooperative launch, with no
// grid barrier: every exchange between CTAs goes through flag-carrying words.
//
// A flag-carrying word is 64 bits: the high half is an epoch (token and layer),
// the low half an fp32 value.  A writer puts the pair with one 64-bit atomic
// exchange; a reader polls the word itself until the epoch is the one it
// expects.  A 64-bit access is single-copy atomic, so a reader never sees a
// value of one epoch with the flag of another, and no fence or counter is
// needed: the time from a write to its use is one L2 round trip.
//
// One CTA per SM: sixteen compute warps and one producer warp.  Per layer and CTA:
//   1. gather r_l (H words; x at layer 0), RMSNorm, quantise h into int16 planes;
//   2. native layers: this CTA's router rows -> logit words; gather all E
//      logits and route them locally (every CTA takes the same decision);
//   3. gate/up: this CTA's slice of the layer's a-values (the K routed experts
//      and the shared expert concatenated, I each): a = silu(G h) * (U h) ->
//      a-words.  LoRA of the shared expert: CTAs 0..2r-1 first publish
//      z_g = A_g h and z_u = A_u h (one row each); the CTAs holding shared
//      rows wait for them, finish a_s = silu(g + s B_g z_g) * (u + s B_u z_u)
//      for their rows and publish partial sums of z_d = A_d a_s over them;
//   4. gather every a-word (and the z_d partial sums);
//   5. down: this CTA's output rows over all of the layer's a-values (lane =
//      output row, warps = half-group units, one cross-warp sum), with the
//      routing weights, the shared expert and s B_d z_d; r_{l+1} = r_l + y ->
//      residual words (r_out at the last layer);
//   6. prerouter head work, off the critical path: fc1 / linear-residual rows
//      of owner l (in the wait for step 4) and fc2 rows of owner l-1 (after
//      step 5), their sums published in the next layer, and at the end of the
//      launch the routing of every head whose logits were completed in it.
//
// Weights reach shared memory by bulk copies (TMA) completing on mbarriers,
// issued by the producer warp a layer ahead where the routing is known (a consumer
// layer routes with the prediction made one token earlier, so its experts
// are known when the token starts), else right after the routing; the
// weights of layer l + D are also prefetched into L2 at the top of layer l.
//
// Every wait is bounded: a thread that gives up raises E0_ST_TIMEOUT and a
// launch-wide abort flag, and its block leaves at its next checked barrier
// (__syncthreads_or of the threads' give-up marks) after waiting for the bulk
// copies it has in flight; every other CTA's polls see the flag and give up
// too.  No CTA touches another CTA's shared memory.
//
// Included inside namespace e0 of e0_decode.cu (StackHdr, LayerP, route_warp).
#pragma once

constexpr int LL_NW = 16;                   // compute warps
constexpr int LL_THREADS = (LL_NW + 1) * 32;  // and one producer warp (bulk copies, L2 prefetch)
constexpr int LL_MAXA = 2;          // a-value passes per warp
constexpr int LL_MAXQ = 10;         // a-words gathered per lane (at most 160 half-group units a layer)
constexpr int LL_MAXB1 = 3;         // fc1 / linear-residual chunks per warp
constexpr int LL_MAXROWS = 16;      // head rows of one CTA; down rows of one CTA
constexpr int LL_RANK = 16;         // largest LoRA rank of this kernel
constexpr int LL_MAX_SHCTA = 64;    // CTAs holding shared-expert rows
constexpr int LL_PF_DIST = 0;       // layers prefetched ahead into L2 (the bulk copies run a layer ahead)
constexpr int LL_MAX_RITEMS = 64;   // router (row, 256-column chunk) items of one CTA

// ------------------------------------------------------------------ flag-carrying words

// The word is written with a relaxed atomic exchange (old value unused)
// rather than a relaxed store: an atomic is carried out at the word's home in
// L2, where the polling readers look, and the 40-layer token ran 8 % faster
// with it (628 against 684 us on one GB300).
E0_DEV void ll_put(unsigned long long* p, float v, uint32_t ep) {
    const unsigned long long w = ((unsigned long long)ep << 32) | (unsigned long long)__float_as_uint(v);
    unsigned long long old;
    asm volatile("atom.relaxed.gpu.global.exch.b64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(w) : "memory");
    (void)old;
}
E0_DEV unsigned long long ll_get(const unsigned long long* p) {
    unsigned long long w;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}
E0_DEV bool ll_ok(unsigned long long w, uint32_t ep) { return (uint32_t)(w >> 32) == ep; }
E0_DEV float ll_val(unsigned long long w) { return __uint_as_float((uint32_t)w); }

// A poll gives up after this much device time by default (a layer takes
// microseconds); e0_stack_prepare may set another limit.
constexpr unsigned long long LL_WAIT_NS = 200000000ull;

struct LLCtx {
    unsigned long long wait_ns;
    unsigned* abort_flag;  // launch-wide (global)
    int* bad;              // this thread's: it gave up (the block leaves at its next __syncthreads_or)
    uint32_t* st;          // status word
};

// Poll until the word carries epoch ep.  Gives up after cx.wait_ns, or as
// soon as another CTA has given up; a thread that gives up returns 0.0 and
// marks itself (the block tests the marks with __syncthreads_or and leaves
// together).
E0_DEV unsigned long long ll_poll(const unsigned long long* p, uint32_t ep, LLCtx cx) {
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (uint32_t it = 1;; ++it) {
        const unsigned long long w = ll_get(p);
        if (ll_ok(w, ep)) return w;
        if ((it & 7u) == 0) {  // each round is an L2 round trip: the clock is read every few
            unsigned ab;
            asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(ab) : "l"(cx.abort_flag) : "memory");
            uint64_t t1;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
            if (ab || t1 - t0 > cx.wait_ns) {
                if (!ab) {
                    atomicExch(cx.abort_flag, 1u);
                    set_status(cx.st, E0_ST_TIMEOUT);
                }
                *cx.bad = 1;
                return (unsigned long long)ep << 32;
            }
        }
    }
}
E0_DEV float ll_take(unsigned long long w, const unsigned long long* p, uint32_t ep, LLCtx cx) {
    if (!ll_ok(w, ep)) w = ll_poll(p, ep, cx);
    return ll_val(w);
}
E0_DEV float ll_wait(const unsigned long long* p, uint32_t ep, LLCtx cx) { return ll_take(ll_get(p), p, ep, cx); }

// Bulk prefetch of [p, p + bytes) into L2: the 16-byte-aligned part inside
// the range (a hint, nothing waits for it).
E0_DEV void l2_prefetch(const void* p, size_t bytes) {
    if (!p || bytes == 0) return;
    uintptr_t a = reinterpret_cast<uintptr_t>(p);
    uintptr_t b = a + bytes;
    a = (a + 15) & ~(uintptr_t)15;
    b &= ~(uintptr_t)15;
    while (b > a) {
        const uintptr_t n = (b - a) > (1u << 30) ? (1u << 30) : (b - a);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"((uint32_t)n) : "memory");
        a += n;
    }
}

E0_DEV int ll_split(int n, int c, int nb) { return (int)((long)n * c / nb); }


// ------------------------------------------------------------------ layer shape

// The layer shape is a compile-time constant of the kernel: H, I, E, K and
// what follows from them (64-groups of H, half-groups and groups of I, rows
// of a warp pass, 256-column chunks of H).
template <int H_, int I_, int E_, int K_>
struct LLShape {
    static constexpr int H = H_, I = I_, E = E_, K = K_;
    static constexpr int GH = H / GROUP, HG = I / 32, GI = I / GROUP;
    static constexpr int G = GH, R = GH >= 32 ? 1 : 32 / GH, NC = H / 256;
    static constexpr int NUm = (K + 1) * I / 32;  // half-group units of a layer with a shared expert
    static constexpr int MAXM = (E + 31) / 32;     // routing scores a lane holds
};

// ------------------------------------------------------------------ per-layer work split

struct LLPart {
    int nk, NAr, NA, NU, A0, A1, J0, J1, Q0, Q1, F0, F1, E0, E1;
    int ps0;       // this CTA's first shared-expert a-value (A1 when it holds none)
    int sh0, nsh;  // first CTA holding shared-expert a-values, and how many do
    bool sh, lora, head, head_prev;
};

// head: this layer owns a head whose prediction feeds a layer; head_prev:
// layer l-1 owns one (its fc2 rows are done during layer l).  Output rows are
// split in the slot layout's blocks of DROWS rows (a block's down codes and
// words are two contiguous ranges).
template <class C>
E0_DEV LLPart ll_part(const LayerP* lyr, int Lz, int l, int c, int nb) {
    LLPart P;
    const LayerP& L = lyr[l];
    P.sh = L.sh != nullptr;
    P.lora = P.sh && L.Ag != nullptr;
    P.nk = C::K + (P.sh ? 1 : 0);
    P.NAr = C::K * C::I;
    P.NA = P.nk * C::I;
    P.NU = P.NA / 32;
    P.A0 = ll_split(P.NA, c, nb);
    P.A1 = ll_split(P.NA, c + 1, nb);
    P.J0 = DROWS * ll_split(C::H / DROWS, c, nb);
    P.J1 = DROWS * ll_split(C::H / DROWS, c + 1, nb);
    P.head = L.fc1 != nullptr && l + 1 < Lz;
    const int nq = P.head ? L.hidden + C::E : 0;
    P.Q0 = ll_split(nq, c, nb);
    P.Q1 = ll_split(nq, c + 1, nb);
    P.head_prev = l >= 1 && lyr[l - 1].fc1 != nullptr;
    const int nf = P.head_prev ? C::E : 0;
    P.F0 = ll_split(nf, c, nb);
    P.F1 = ll_split(nf, c + 1, nb);
    P.E0 = ll_split(C::E, c, nb);
    P.E1 = ll_split(C::E, c + 1, nb);
    P.ps0 = P.A1;
    P.sh0 = nb;
    P.nsh = 0;
    if (P.sh) {
        P.ps0 = max(P.A0, P.NAr);
        if (P.ps0 > P.A1) P.ps0 = P.A1;
        // the shared expert is the last one: its a-values belong to CTAs sh0..nb-1
        int s0 = (int)((long)P.NAr * nb / P.NA);
        s0 = s0 > 1 ? s0 - 1 : 0;
        while (s0 < nb && ll_split(P.NA, s0 + 1, nb) <= P.NAr) ++s0;
        P.sh0 = s0;
        P.nsh = nb - s0;
    }
    return P;
}

// ------------------------------------------------------------------ shared memory

// Per-launch maxima of the work split (the same on host and device).
struct LLGeo {
    int ma, mq, me, mf, nr;
    __host__ __device__ LLGeo(int H, int I, int E, int K, int hidden, int nb) {
        auto cdiv = [](long a, long b) { return (int)((a + b - 1) / b); };
        ma = cdiv((long)(K + 1) * I, nb);
        mq = cdiv((long)hidden + E, nb);
        me = cdiv(E, nb);
        mf = cdiv(E, nb);
        nr = DROWS * cdiv(H / DROWS, nb);
    }
};

struct LLSmem {
    uint32_t hdr, lyr, r, hpl, hxg, red, inds, w, prev, slots, tab, lg, scr, apl, axg, pb1, poh, pb2, prt, pla, ghp,
        ypart, zv, aso, zdp, bars;
    // staging of bulk copies: head-side buffers (two, by layer parity), gate/up, down
    uint32_t hbuf[2], h_la, h_f2, h_bd, h_rt, h_bytes;
    uint32_t g_codes, g_sb, g_bg, g_bu, g_rows, d_codes, d_sb;
    uint32_t total;
    __host__ __device__ LLSmem(int H, int I, int E, int L, int K, int hidden, int nb) {
        const LLGeo g(H, I, E, K, hidden, nb);
        const int GH = H / GROUP;
        const int NUm = (K + 1) * I / 32;
        size_t o = 0;
        auto take = [&](size_t n) {
            const size_t at = o;
            o = (o + n + 15) & ~(size_t)15;
            return (uint32_t)at;
        };
        // regions whose size follows from the layer shape alone come first: in
        // the kernel their offsets are compile-time constants
        hdr = take(sizeof(StackHdr));
        r = take((size_t)H * 4);
        hpl = take((size_t)GH * 8 * 16);
        hxg = take((size_t)GH * sizeof(XGroup));
        red = take(32 * 4);
        tab = take((size_t)E * 4);
        lg = take((size_t)E * 4);
        scr = take((size_t)2 * E * 4);
        apl = take((size_t)NUm * 4 * 16);
        axg = take((size_t)NUm * sizeof(XGroup));
        pb1 = take((size_t)2 * LL_MAXB1 * LL_NW * 4);  // head partial sums, by layer parity
        poh = take(2 * LL_MAXROWS * 4);
        pb2 = take(2 * LL_NW * 4);
        prt = take(LL_MAX_RITEMS * 4);
        pla = take(LL_NW * 4);
        ypart = take((size_t)2 * LL_NW * LL_MAXROWS * 4);
        zv = take(3 * LL_RANK * 4);
        zdp = take((size_t)LL_MAX_SHCTA * LL_RANK * 4);
        bars = take(4 * 8);  // head-side [2], gate/up, down
        // then those sized by the layer count, the head width and the grid
        lyr = take((size_t)L * sizeof(LayerP));
        inds = take((size_t)L * K * 4);
        w = take((size_t)L * K * 4);
        prev = take((size_t)L * K * 4);
        slots = take((size_t)L * (K + 1) * 8);
        ghp = take((size_t)(hidden > 0 ? hidden : 1) * 4);
        aso = take((size_t)g.ma * 4);
        // head-side buffer (two, by layer parity): LoRA A row, fc2 rows, B_down rows, router rows
        size_t hb = 0;
        h_la = (uint32_t)hb;
        hb += (size_t)H * 2;
        h_f2 = (uint32_t)hb;
        hb += (size_t)g.mf * (hidden > 0 ? hidden : 1) * 2;
        hb = (hb + 15) & ~(size_t)15;
        h_bd = (uint32_t)hb;
        hb += (size_t)g.nr * LL_RANK * 2;
        h_rt = (uint32_t)hb;
        hb += (size_t)g.me * H * 2;
        h_bytes = (uint32_t)((hb + 127) & ~(size_t)127);
        o = (o + 127) & ~(size_t)127;
        hbuf[0] = take(h_bytes);
        hbuf[1] = take(h_bytes);
        // gate/up side: gate/up rows, their (scale, bias) words, B_gate / B_up
        // rows, and the head rows of the layer's owner
        g_codes = take((size_t)g.ma * H);
        g_sb = take((size_t)g.ma * 2 * GH * 4);
        g_bg = take((size_t)g.ma * LL_RANK * 2);
        g_bu = take((size_t)g.ma * LL_RANK * 2);
        g_rows = take((size_t)g.mq * H * 2);
        // down side, per expert: this CTA's row blocks, [block][half-group][row
        // in block][16 code bytes] and [block][64-group][row in block] words
        d_codes = take((size_t)(K + 1) * (I / 32) * g.nr * 16);
        d_sb = take((size_t)(K + 1) * (I / GROUP) * g.nr * 4);
        total = (uint32_t)((o + 127) & ~(size_t)127);
    }
};

// ------------------------------------------------------------------ bulk copies and mbarriers

E0_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
E0_DEV void ll_mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
E0_DEV void ll_mbar_expect(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// weights are read once from HBM: evict-first in L2
E0_DEV void ll_bulk(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(l2_evict_first())
        : "memory");
}
// Bounded wait for phase `parity` of an mbarrier (false: gave up).  The
// waiting thread is suspended in try_wait (up to a microsecond a try) rather
// than spinning, so waiting warps leave the issue slots to the others.
E0_DEV bool ll_mbar_wait(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
    const uint32_t a = smem_u32(bar);
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(a), "r"(parity), "r"(1000u)
            : "memory");
        if (ok) return true;
        uint64_t t1;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
        if (it == 0) t0 = t1;
        else if (t1 - t0 > limit_ns) return false;
    }
}

// One warp issues a list of bulk copies completing on `bar` (one arrival with
// the total bytes, made before the copies).  item(i, dst, src, bytes) gives
// copy i (bytes 0: none).
template <class Item>
E0_DEV void ll_issue(uint64_t* bar, int n, Item item, int lane) {
    uint32_t tot = 0;
    for (int i = lane; i < n; i += 32) {
        void* d = nullptr;
        const void* s = nullptr;
        uint32_t b = 0;
        item(i, d, s, b);
        tot += b;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    // the buffers were last read through the generic proxy (ordered by the
    // block barrier that precedes every issue)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) ll_mbar_expect(bar, tot);
    __syncwarp();
    for (int i = lane; i < n; i += 32) {
        void* d = nullptr;
        const void* s = nullptr;
        uint32_t b = 0;
        item(i, d, s, b);
        if (b) ll_bulk(d, s, b, bar);
    }
}

// ------------------------------------------------------------------ L2 prefetch of one layer

// This CTA's share of layer m's weights: its 1/nb byte slice of each expert
// slot the layer reads (routed ones only when `routed` is set), its head
// rows (first H columns), its fc2 rows of owner m-1, its router rows (native
// layers), and its 1/nb slices of the LoRA matrices.  One warp.
template <class C>
E0_DEV void ll_prefetch_layer(const LayerP* lyr, int Lz, const uint8_t* const* slots, int m, bool native, bool routed,
                              bool only_routed, int c, int nb, int lane) {
    const LayerP& L = lyr[m];
    const LLPart P = ll_part<C>(lyr, Lz, m, c, nb);
    constexpr int K = C::K, H = C::H, E = C::E;
    const size_t SB = SlotLayout{H, C::I}.bytes();
    const size_t s0 = (size_t)ll_split((int)(SB / 16), c, nb) * 16, s1 = (size_t)ll_split((int)(SB / 16), c + 1, nb) * 16;
    const size_t ld = (size_t)H + 2 * E;
    const int nrow = P.Q1 - P.Q0;
    const int n_items = only_routed ? K : (K + 1) + 2 + nrow + 6;
    for (int i = lane; i < n_items; i += 32) {
        const void* p = nullptr;
        size_t n = 0;
        if (i <= K) {
            if (i < K ? routed : true) {
                const uint8_t* ex = slots[(size_t)m * (K + 1) + i];
                if (ex) {
                    p = ex + s0;
                    n = s1 - s0;
                }
            }
        } else if (i == K + 1) {
            if (native && L.W_r) {
                p = L.W_r + (size_t)P.E0 * H;
                n = (size_t)(P.E1 - P.E0) * H * 2;
            }
        } else if (i == K + 2) {
            if (P.head_prev) {
                const LayerP& O = lyr[m - 1];
                p = O.fc2 + (size_t)P.F0 * O.hidden;
                n = (size_t)(P.F1 - P.F0) * O.hidden * 2;
            }
        } else if (i < K + 3 + nrow) {
            const int q = P.Q0 + (i - K - 3);
            p = q < L.hidden ? L.fc1 + (size_t)q * ld : L.lres + (size_t)(q - L.hidden) * ld;
            n = (size_t)H * 2;
        } else if (P.lora) {
            const int j = i - K - 3 - nrow, R = L.rank;
            const __half* mats[6] = {L.Ag, L.Au, L.Bg, L.Bu, L.Ad, L.Bd};
            const size_t el[6] = {(size_t)R * H, (size_t)R * H, (size_t)C::I * R, (size_t)C::I * R, (size_t)R * C::I,
                                  (size_t)H * R};
            const size_t units = el[j] * 2 / 16;
            const size_t a = units * c / nb * 16, b = units * (c + 1) / nb * 16;
            p = reinterpret_cast<const uint8_t*>(mats[j]) + a;
            n = b - a;
        }
        l2_prefetch(p, n);
    }
}



// ------------------------------------------------------------------ the kernel

template <class C>
__global__ void __launch_bounds__(LL_THREADS, 1)
    k_stack_ll(StackHdr* Sp, const float* x, float* r_out, TraceP tr, uint32_t* st, int lb, int le) {
    constexpr int H = C::H, I = C::I, E = C::E, K = C::K;
    constexpr int GH = C::GH, HG = C::HG, GI = C::GI, G = C::G, R = C::R, NC = C::NC;
    constexpr int PROD = LL_NW;  // the producer warp
    extern __shared__ __align__(128) char smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool cw = warp < LL_NW;  // a compute warp
    const int nb = gridDim.x, c = blockIdx.x;
    const int Lz = Sp->L;
    const LLSmem lay(H, I, E, Lz, K, Sp->hidden, nb);
    {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(Sp);
        uint32_t* dst = reinterpret_cast<uint32_t*>(smem + lay.hdr);
        for (int i = tid; i < (int)(sizeof(StackHdr) / 4); i += LL_THREADS) dst[i] = src[i];
        const uint32_t* ls = reinterpret_cast<const uint32_t*>(Sp->layers);
        uint32_t* ldp = reinterpret_cast<uint32_t*>(smem + lay.lyr);
        for (int i = tid; i < (int)((size_t)Lz * sizeof(LayerP) / 4); i += LL_THREADS) ldp[i] = ls[i];
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);  // head-side [2], gate/up, down
    if (tid == 0) {
        for (int b = 0; b < 4; ++b) ll_mbar_init(&bars[b], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const StackHdr& S = *reinterpret_cast<const StackHdr*>(smem + lay.hdr);
    const LayerP* lyr = reinterpret_cast<const LayerP*>(smem + lay.lyr);
    const int t = S.t;
    const uint32_t ep0 = (uint32_t)t * (uint32_t)Lz + 1u;  // epoch of layer l: ep0 + l
    const SlotLayout sl{H, I};
    const size_t SB = sl.bytes(), gusb = sl.gu_sb(), dcode = sl.down_codes(), dsbo = sl.down_sb();
    const size_t ldh = (size_t)H + 2 * E;  // row length of head fc1 / linear residual
    const int pf_dist = S.pf_dist;
    const unsigned long long wait_ns = S.ll_wait_ns;

    float* r = reinterpret_cast<float*>(smem + lay.r);
    uint4* hpl = reinterpret_cast<uint4*>(smem + lay.hpl);
    XGroup* hxg = reinterpret_cast<XGroup*>(smem + lay.hxg);
    float* red = reinterpret_cast<float*>(smem + lay.red);
    int32_t* inds_s = reinterpret_cast<int32_t*>(smem + lay.inds);
    float* w_s = reinterpret_cast<float*>(smem + lay.w);
    int32_t* prev_s = reinterpret_cast<int32_t*>(smem + lay.prev);
    const uint8_t** slot_s = reinterpret_cast<const uint8_t**>(smem + lay.slots);
    int32_t* tab_s = reinterpret_cast<int32_t*>(smem + lay.tab);
    float* lg = reinterpret_cast<float*>(smem + lay.lg);
    float* scr = reinterpret_cast<float*>(smem + lay.scr);
    uint4* apl = reinterpret_cast<uint4*>(smem + lay.apl);
    XGroup* axg = reinterpret_cast<XGroup*>(smem + lay.axg);
    float* pb1 = reinterpret_cast<float*>(smem + lay.pb1);
    float* poh = reinterpret_cast<float*>(smem + lay.poh);
    float* pb2 = reinterpret_cast<float*>(smem + lay.pb2);
    float* prt = reinterpret_cast<float*>(smem + lay.prt);
    float* pla = reinterpret_cast<float*>(smem + lay.pla);
    float* ghp = reinterpret_cast<float*>(smem + lay.ghp);  // gelu of owner l-1's hidden words
    float* ypart = reinterpret_cast<float*>(smem + lay.ypart);
    float* zv = reinterpret_cast<float*>(smem + lay.zv);    // z_d at [2 LL_RANK ..]
    float* aso = reinterpret_cast<float*>(smem + lay.aso);  // this CTA's finished shared a-values
    float* zdp = reinterpret_cast<float*>(smem + lay.zdp);  // gathered partial sums of z_d
    auto hbuf = [&](int l) { return smem + lay.hbuf[0] + (size_t)(l & 1) * (lay.hbuf[1] - lay.hbuf[0]); };
    char* gcodes = smem + lay.g_codes;
    char* gsb = smem + lay.g_sb;
    const __half* gbg = reinterpret_cast<const __half*>(smem + lay.g_bg);
    const __half* gbu = reinterpret_cast<const __half*>(smem + lay.g_bu);
    char* dcodes = smem + lay.d_codes;
    char* dsb = smem + lay.d_sb;
    int bad = 0;
    const LLCtx cx{wait_ns, &Sp->ll_abort, &bad, st};
    uint32_t* st0 = c == 0 ? st : nullptr;
    // bulk-copy phases issued (producer) and waited (compute warps) on each mbarrier
    int iss_h0 = 0, iss_h1 = 0, iss_g = 0, iss_d = 0;
    int wt_h0 = 0, wt_h1 = 0, wt_g = 0, wt_d = 0;
    auto wait_bar = [&](uint64_t* bar, int& w) {
        if (!ll_mbar_wait(bar, (uint32_t)(w & 1), wait_ns)) {
            bad = 1;
            set_status(st, E0_ST_TIMEOUT);
        }
        ++w;
    };
    // before the block leaves: the bulk copies it issued have landed
    auto leave = [&]() {
        if (warp == PROD && lane == 0) {
            if (iss_h0) ll_mbar_wait(&bars[0], (uint32_t)((iss_h0 - 1) & 1), 1000000000ull);
            if (iss_h1) ll_mbar_wait(&bars[1], (uint32_t)((iss_h1 - 1) & 1), 1000000000ull);
            if (iss_g) ll_mbar_wait(&bars[2], (uint32_t)((iss_g - 1) & 1), 1000000000ull);
            if (iss_d) ll_mbar_wait(&bars[3], (uint32_t)((iss_d - 1) & 1), 1000000000ull);
        }
    };

    // routing known when the token starts (consumer layers take the prediction
    // made one token earlier) and the previous token's routing (head input)
    for (int q = tid; q < Lz * K; q += LL_THREADS) {
        const int l = q / K, k = q % K;
        prev_s[q] = t > 0 ? __ldcg(S.hist + ((size_t)((t + 1) & 1) * Lz + l) * K + k) : -1;
        inds_s[q] = -1;
        w_s[q] = 0.f;
        if (!layer_native(S, lyr[l], t)) {
            const size_t o = ((size_t)(t & 1) * Lz + l) * K + k;
            inds_s[q] = __ldcg(S.pred_inds + o);
            w_s[q] = __ldcg(S.pred_w + o);
        }
    }
    __syncthreads();
    for (int q = tid; q < Lz * (K + 1); q += LL_THREADS) {
        const int l = q / (K + 1), k = q % (K + 1);
        const LayerP& L = lyr[l];
        if (k == K) {
            slot_s[q] = L.sh;
            continue;
        }
        slot_s[q] = nullptr;
        if (!layer_native(S, L, t)) {
            const int e = inds_s[l * K + k];
            const int s2 = (e >= 0 && e < E) ? __ldcg(L.table + e) : -1;
            slot_s[q] = (s2 >= 0 && s2 < L.n_slots) ? L.pool + (size_t)s2 * SB : nullptr;
        }
    }
    __syncthreads();

    // ---- bulk copies of one layer (the producer warp issues them)
    // head side (buffer l & 1): LoRA A row, fc2 rows of owner l-1, B_down
    // rows, router rows (native layers)
    auto issue_h = [&](int l) {
        const LayerP& L = lyr[l];
        const LLPart P = ll_part<C>(lyr, Lz, l, c, nb);
        char* b = hbuf(l);
        const int rk = P.lora ? L.rank : 0;
        const bool nat = layer_native(S, L, t);
        auto item = [&](int i, void*& d, const void*& s, uint32_t& n) {
            if (i == 0) {
                if (P.lora && c < 2 * rk) {
                    d = b + lay.h_la;
                    s = c < rk ? L.Ag + (size_t)c * H : L.Au + (size_t)(c - rk) * H;
                    n = (uint32_t)H * 2;
                }
            } else if (i == 1) {
                if (P.head_prev && P.F1 > P.F0) {
                    const LayerP& O = lyr[l - 1];
                    d = b + lay.h_f2;
                    s = O.fc2 + (size_t)P.F0 * O.hidden;
                    n = (uint32_t)(P.F1 - P.F0) * O.hidden * 2;
                }
            } else if (i == 2) {
                if (P.lora && P.J1 > P.J0) {
                    d = b + lay.h_bd;
                    s = L.Bd + (size_t)P.J0 * rk;
                    n = (uint32_t)(P.J1 - P.J0) * rk * 2;
                }
            } else if (nat && L.W_r && P.E1 > P.E0) {
                d = b + lay.h_rt;
                s = L.W_r + (size_t)P.E0 * H;
                n = (uint32_t)(P.E1 - P.E0) * H * 2;
            }
        };
        ll_issue(&bars[l & 1], 4, item, lane);
        if (l & 1) ++iss_h1;
        else ++iss_h0;
    };
    // gate/up side: this CTA's gate/up rows (codes, (scale, bias) words), for
    // shared-expert rows with LoRA their B_gate / B_up rows, and this CTA's
    // head rows of owner l (first H columns)
    auto issue_g = [&](int l) {
        const LayerP& L = lyr[l];
        const LLPart P = ll_part<C>(lyr, Lz, l, c, nb);
        const uint8_t* const* sq = slot_s + (size_t)l * (K + 1);
        const int rk = P.lora ? L.rank : 0;
        const int q0 = P.A1 > P.A0 ? P.A0 / I : 0, q1 = P.A1 > P.A0 ? (P.A1 - 1) / I + 1 : 0;
        const int nrun = q1 - q0;
        auto item = [&](int i, void*& d, const void*& s, uint32_t& n) {
            if (i < 2 * nrun) {
                const int q = q0 + i / 2;
                const int p0 = max(P.A0, q * I), p1 = min(P.A1, (q + 1) * I);
                const uint8_t* ex = sq[q];
                if (!ex || p1 <= p0) return;
                if ((i & 1) == 0) {
                    d = gcodes + (size_t)(p0 - P.A0) * H;
                    s = ex + (size_t)(p0 - q * I) * H;
                    n = (uint32_t)(p1 - p0) * H;
                } else {
                    d = gsb + (size_t)(p0 - P.A0) * 2 * GH * 4;
                    s = ex + gusb + (size_t)(p0 - q * I) * 2 * GH * 4;
                    n = (uint32_t)(p1 - p0) * 2 * GH * 4;
                }
            } else if (i < 2 * nrun + 2) {
                if (P.lora && P.A1 > P.ps0) {
                    const int i0 = P.ps0 - P.NAr, cnt = P.A1 - P.ps0;
                    d = smem + (i == 2 * nrun ? lay.g_bg : lay.g_bu);
                    s = (i == 2 * nrun ? L.Bg : L.Bu) + (size_t)i0 * rk;
                    n = (uint32_t)cnt * rk * 2;
                }
            } else {
                const int k = i - 2 * nrun - 2, q = P.Q0 + k;
                d = smem + lay.g_rows + (size_t)k * H * 2;
                s = q < L.hidden ? L.fc1 + (size_t)q * ldh : L.lres + (size_t)(q - L.hidden) * ldh;
                n = (uint32_t)H * 2;
            }
        };
        ll_issue(&bars[2], 2 * nrun + 2 + (P.Q1 - P.Q0), item, lane);
        ++iss_g;
    };
    // down side: per expert, this CTA's row blocks of down codes (every input)
    // and of their (scale, bias) words, two contiguous ranges
    const int NRM = DROWS;  // rows of a down block (a CTA takes one block or none)
    auto issue_d = [&](int l) {
        const LLPart P = ll_part<C>(lyr, Lz, l, c, nb);
        const uint8_t* const* sq = slot_s + (size_t)l * (K + 1);
        const size_t bcb = sl.down_block_code_bytes(), bsb = sl.down_block_sb_bytes();
        const int blk = P.J0 / DROWS;
        auto item = [&](int i, void*& d, const void*& s, uint32_t& n) {
            if (P.J1 <= P.J0) return;
            const int q = i % P.nk;
            const uint8_t* ex = sq[q];
            if (!ex) return;
            if (i < P.nk) {
                d = dcodes + (size_t)q * bcb;
                s = ex + dcode + (size_t)blk * bcb;
                n = (uint32_t)bcb;
            } else {
                d = dsb + (size_t)q * bsb;
                s = ex + dsbo + (size_t)blk * bsb;
                n = (uint32_t)bsb;
            }
        };
        ll_issue(&bars[3], 2 * P.nk, item, lane);
        ++iss_d;
    };

    if (warp == PROD) {
        issue_h(lb);
        if (!layer_native(S, lyr[lb], t)) {
            issue_g(lb);
            issue_d(lb);
        }
        for (int m = lb; m < le && m < lb + pf_dist; ++m) {
            const bool nat = layer_native(S, lyr[m], t);
            ll_prefetch_layer<C>(lyr, Lz, slot_s, m, nat, !nat, false, c, nb, lane);
        }
    }

    int pend = -1;  // layer whose head partial sums wait to be published
    // Publish the head sums left by layer lp: fc1 / linear-residual rows of
    // owner lp (hidden and zres words, b1 given per thread), fc2 rows of owner
    // lp-1 (logit words, with b2 and zrv, the zres word of owner lp-1).
    auto combine = [&](int lp, float b1v, float b2v, float zrv) {
        const LLPart P = ll_part<C>(lyr, Lz, lp, c, nb);
        const LayerP& L = lyr[lp];
        const int pp = lp & 1;  // partial sums of layer lp (double-buffered: the next layer writes the other half)
        if (P.head && tid < P.Q1 - P.Q0) {
            const int hid = L.hidden, q = P.Q0 + tid;
            unsigned long long* hpw = S.llHp + (size_t)(lp & 1) * (hid + E);
            float v = poh[pp * LL_MAXROWS + tid] + b1v;
            for (int ch = 0; ch < NC; ++ch) v += pb1[pp * LL_MAXB1 * LL_NW + tid * NC + ch];
            ll_put(hpw + q, v, ep0 + lp);
        }
        if (P.head_prev && tid >= 32 && tid - 32 < P.F1 - P.F0) {
            const LayerP& O = lyr[lp - 1];
            const int NCF = O.hidden / 256, e0 = tid - 32, e = P.F0 + e0;
            float v = b2v + zrv;
            for (int ch = 0; ch < NCF; ++ch) v += pb2[pp * LL_NW + e0 * NCF + ch];
            ll_put(S.llZ + (size_t)(lp - 1) * E + e, v, ep0 + lp);
            if (tr.head_logits) tr.head_logits[(size_t)(lp - 1) * E + e] = v;
        }
    };
    // this thread's bias terms for combine(lp), as raw fp16 bits (converted at use)
    auto combine_bias = [&](int lp, unsigned short& b1h, unsigned short& b2h) {
        b1h = b2h = 0;
        const LLPart P = ll_part<C>(lyr, Lz, lp, c, nb);
        const LayerP& L = lyr[lp];
        if (P.head && tid < P.Q1 - P.Q0 && P.Q0 + tid < L.hidden && L.b1)
            b1h = __ldg(reinterpret_cast<const unsigned short*>(L.b1) + P.Q0 + tid);
        if (P.head_prev && tid >= 32 && tid - 32 < P.F1 - P.F0 && lyr[lp - 1].b2)
            b2h = __ldg(reinterpret_cast<const unsigned short*>(lyr[lp - 1].b2) + P.F0 + tid - 32);
    };
    auto h2f = [](unsigned short h) { return __half2float(__ushort_as_half(h)); };
    // The zres word of owner lp-1 that this thread's fc2 row adds in
    // combine(lp) (null: none).  It must be read before this CTA publishes an
    // a-word of layer lp+1: until then no CTA can finish that layer and rewrite
    // the word's buffer (owner lp+1's words, two layers on), whether or not
    // this CTA holds down rows.
    auto zres_word = [&](int lp) -> const unsigned long long* {
        const LLPart P = ll_part<C>(lyr, Lz, lp, c, nb);
        if (!(P.head_prev && tid >= 32 && tid - 32 < P.F1 - P.F0)) return nullptr;
        const LayerP& O = lyr[lp - 1];
        return S.llHp + (size_t)((lp - 1) & 1) * (O.hidden + E) + O.hidden + P.F0 + (tid - 32);
    };

    for (int l = lb; l < le; ++l) {
        const LayerP& L = lyr[l];
        const bool native = layer_native(S, L, t);
        const LLPart P = ll_part<C>(lyr, Lz, l, c, nb);
        const uint32_t ep = ep0 + l;
        const uint8_t* const* sl_l = slot_s + (size_t)l * (K + 1);
        const int rank = P.lora ? L.rank : 0;
        int32_t* inds = inds_s + (size_t)l * K;
        float* wts = w_s + (size_t)l * K;
        const int nq = P.Q1 - P.Q0;
        const int nb1 = P.head ? nq * NC : 0;
        const int NR = P.J1 - P.J0;
        char* hb = hbuf(l);
        const int lp = pend;  // the head sums of the previous layer are published in this one
        const int n_own = P.A1 - P.ps0;  // this CTA's shared-expert a-values
        unsigned short b1h = 0, b2h = 0, adh = 0, ohh = 0;
        int tabv0 = -1, tabv1 = -1;
        const unsigned long long* zrp = nullptr;  // the zres word of combine(lp)
        unsigned long long zrw = 0;
        // the one-hot terms of this layer's head rows (lane < 2K of warp q - Q0):
        // this layer's experts, then the previous token's
        auto load_oh = [&]() {
            if (P.head && warp < nq && lane < 2 * K) {
                const int q = P.Q0 + warp;
                const __half* row = q < L.hidden ? L.fc1 + (size_t)q * ldh : L.lres + (size_t)(q - L.hidden) * ldh;
                const int e = lane < K ? inds[lane] : prev_s[(size_t)l * K + lane - K];
                if (e >= 0 && e < E)
                    ohh = __ldg(reinterpret_cast<const unsigned short*>(row) + (lane < K ? (size_t)H : (size_t)H + E) + e);
            }
        };

        if (warp == PROD) {
            // ---- prefetch of layer l + D into L2 (D = 0: none; the bulk copies
            // already fetch layer l)
            if (pf_dist > 0 && l + pf_dist < le) {
                const int m = l + pf_dist;
                const bool nat = layer_native(S, lyr[m], t);
                ll_prefetch_layer<C>(lyr, Lz, slot_s, m, nat, !nat, false, c, nb, lane);
            }
        } else {
            // ---- small loads that do not wait for h: the expert table (native),
            // the bias terms of the head sums published in this layer, this CTA's
            // A_down entries (LoRA partial sums), the one-hot terms
            if (native) {
                if (tid < E) tabv0 = __ldcg(L.table + tid);
                if (tid + LL_NW * 32 < E) tabv1 = __ldcg(L.table + tid + LL_NW * 32);
            }
            if (lp >= 0) {
                combine_bias(lp, b1h, b2h);
                zrp = zres_word(lp);
                if (zrp) zrw = ll_get(zrp);  // in flight with the residual words below
            }
            if (P.lora && warp < rank && lane < n_own)
                adh = __ldg(reinterpret_cast<const unsigned short*>(L.Ad) + (size_t)warp * I + (P.ps0 - P.NAr) + lane);
            if (!native) load_oh();

            // ---- 1. r_l, RMSNorm statistics, quantised planes of h (of r: the codes
            // of a group do not change with its scale; products are scaled by
            // inv_denom afterwards)
            float ss = 0.f;
            float2 v0 = make_float2(0.f, 0.f), v1 = make_float2(0.f, 0.f);
            unsigned long long wa0 = 0, wb0 = 0, wa1 = 0, wb1 = 0;
            const int g0 = warp, g1 = warp + LL_NW;
            const int j0 = GROUP * g0 + 2 * lane, j1 = GROUP * g1 + 2 * lane;
            if (l == 0) {
                if (g0 < GH) v0 = __ldcg(reinterpret_cast<const float2*>(x + j0));
                if (g1 < GH) v1 = __ldcg(reinterpret_cast<const float2*>(x + j1));
            } else {
                if (g0 < GH) {
                    wa0 = ll_get(S.llR + j0);
                    wb0 = ll_get(S.llR + j0 + 1);
                }
                if (g1 < GH) {
                    wa1 = ll_get(S.llR + j1);
                    wb1 = ll_get(S.llR + j1 + 1);
                }
            }
            if (g0 < GH) {
                if (l > 0) {
                    v0.x = ll_take(wa0, S.llR + j0, ep - 1, cx);
                    v0.y = ll_take(wb0, S.llR + j0 + 1, ep - 1, cx);
                }
                *reinterpret_cast<float2*>(r + j0) = v0;
                ss = fmaf(v0.x, v0.x, fmaf(v0.y, v0.y, ss));
                quantize_group_v(v0, hpl + g0, hxg + g0, lane, st0, GH);
            }
            if (g1 < GH) {
                if (l > 0) {
                    v1.x = ll_take(wa1, S.llR + j1, ep - 1, cx);
                    v1.y = ll_take(wb1, S.llR + j1 + 1, ep - 1, cx);
                }
                *reinterpret_cast<float2*>(r + j1) = v1;
                ss = fmaf(v1.x, v1.x, fmaf(v1.y, v1.y, ss));
                quantize_group_v(v1, hpl + g1, hxg + g1, lane, st0, GH);
            }
            ss = warp_sum(ss);
            if (lane == 0) red[warp] = ss;
            if (native) {
                if (tid < E) tab_s[tid] = tabv0;
                if (tid + LL_NW * 32 < E) tab_s[tid + LL_NW * 32] = tabv1;
            }
            // the zres word, taken before the barrier below (which precedes every
            // a-word this CTA publishes in layer l); kept in the z_d gather area,
            // unused until step 4
            if (zrp) zdp[tid] = ll_take(zrw, zrp, ep0 + lp - 1, cx);
        }
        // a thread that gave up waiting: the whole block leaves
        if (__syncthreads_or(bad)) {
            leave();
            return;
        }
        // the head-side buffer of layer l + 1 was last read by layer l - 1
        if (warp == PROD && l + 1 < le) issue_h(l + 1);
        pend = -1;
        float inv_denom;
        {
            float tot = lane < LL_NW ? red[lane] : 0.f;
            tot = warp_sum(tot);
            inv_denom = 1.f / sqrtf(tot / (float)H + 1e-6f);
        }
        if (c == 0 && tr.r && cw)
            for (int j = tid; j < H; j += LL_NW * 32) tr.r[(size_t)l * H + j] = r[j];
        if (cw) {
            if (l & 1) wait_bar(&bars[1], wt_h1);
            else wait_bar(&bars[0], wt_h0);
        }

        // ---- 2. native routing: router rows -> logit words, gather, route
        if (native) {
            const int nit = (P.E1 - P.E0) * NC;
            if (cw)
                for (int it = warp; it < nit; it += LL_NW) {
                    const int ch = it % NC;
                    const uint4 wv = *reinterpret_cast<const uint4*>(
                        hb + lay.h_rt + ((size_t)(it / NC) * H + ch * 256 + lane * 8) * 2);
                    const float4 a0 = *reinterpret_cast<const float4*>(r + ch * 256 + lane * 8);
                    const float4 a1 = *reinterpret_cast<const float4*>(r + ch * 256 + lane * 8 + 4);
                    const float v = warp_sum(h8_dot44(wv, a0, a1));
                    if (lane == 0) prt[it] = v;
                }
            __syncthreads();
            for (int e0 = tid; e0 < P.E1 - P.E0; e0 += LL_THREADS) {
                float v = 0.f;
                for (int ch = 0; ch < NC; ++ch) v += prt[e0 * NC + ch];
                ll_put(S.llLg + P.E0 + e0, v * inv_denom, ep);
            }
            for (int e = tid; e < E; e += LL_THREADS) lg[e] = ll_wait(S.llLg + e, ep, cx);
            if (__syncthreads_or(bad)) {
                leave();
                return;
            }
            if (warp == 0) route_warp_t<C::MAXM>(lg, E, S.rp, inds, wts, scr, st0, lane);
            __syncthreads();
            if (tid < K) {
                const int e = inds[tid];
                const int s2 = (e >= 0 && e < E) ? tab_s[e] : -1;
                slot_s[(size_t)l * (K + 1) + tid] = (s2 >= 0 && s2 < L.n_slots) ? L.pool + (size_t)s2 * SB : nullptr;
            }
            __syncthreads();
            if (warp == PROD) {
                issue_g(l);
                issue_d(l);
                ll_prefetch_layer<C>(lyr, Lz, slot_s, l, false, true, true, c, nb, lane);
            } else {
                load_oh();
            }
        }
        if (c == 0 && warp == 1 && lane < K) {
            const int e = inds[lane];
            if (!sl_l[lane]) set_status(st, (e < 0 || e >= E) ? E0_ST_BAD_EXPERT : E0_ST_SLOT_MISS);
            S.hist[((size_t)(t & 1) * Lz + l) * K + lane] = e;
            S.wcur[(size_t)l * K + lane] = wts[lane];
            if (tr.inds) tr.inds[(size_t)l * K + lane] = e;
            if (tr.w) tr.w[(size_t)l * K + lane] = wts[lane];
        }

        // ---- 3. gate/up
        const bool la_cta = P.lora && c < 2 * rank;
        float kg0 = 0.f, ku0 = 0.f, kg1 = 0.f, ku1 = 0.f;
        if (cw) {
            // LoRA A rows of the shared expert first (they need only r and the
            // head-side buffer): CTA c < 2r takes row c of [A_gate ; A_up],
            // warps 8..15 one 256-column chunk each
            if (la_cta && warp >= 8) {
                const int ch = warp - 8;
                float v = 0.f;
                if (ch < NC) {
                    const uint4 wv = *reinterpret_cast<const uint4*>(hb + lay.h_la + (size_t)(ch * 256 + lane * 8) * 2);
                    const float4 a0 = *reinterpret_cast<const float4*>(r + ch * 256 + lane * 8);
                    const float4 a1 = *reinterpret_cast<const float4*>(r + ch * 256 + lane * 8 + 4);
                    v = h8_dot44(wv, a0, a1);
                }
                v = warp_sum(v);
                if (lane == 0) pla[warp - 8] = v;
                asm volatile("bar.sync 1, 256;" ::: "memory");
                if (warp == 8 && lane == 0) {
                    float z = 0.f;
                    for (int k = 0; k < 8; ++k) z += pla[k];
                    ll_put(S.llZg + c, z * inv_denom, ep);
                }
            }
            wait_bar(&bars[2], wt_g);
            // this CTA's a-values: a = silu(G h) * (U h) -> a-words; a shared-expert
            // row with LoRA keeps its pre-activations for the LoRA terms below
            const int g = lane % G;
#pragma unroll
            for (int m = 0; m < LL_MAXA; ++m) {
                const int pw = P.A0 + (warp + LL_NW * m) * R;  // first a-value of this warp pass
                if (pw >= P.A1) continue;
                const int p = pw + lane / G;
                const bool live = lane < R * G && p < P.A1;
                const int q = live ? p / I : 0;
                const uint8_t* ex = live ? sl_l[q] : nullptr;
                float pg = 0.f, pu = 0.f;
                if (ex) {
                    const char* cg = gcodes + (size_t)(p - P.A0) * H + 32 * g;
                    const uint32_t* sbw = reinterpret_cast<const uint32_t*>(gsb + (size_t)(p - P.A0) * 2 * GH * 4) + g;
                    pg = q4_group_dot(*reinterpret_cast<const uint4*>(cg), *reinterpret_cast<const uint4*>(cg + 16),
                                      hpl + g, hxg[g], sbw[0], GH);
                    pu = q4_group_dot(*reinterpret_cast<const uint4*>(cg + H / 2),
                                      *reinterpret_cast<const uint4*>(cg + H / 2 + 16), hpl + g, hxg[g], sbw[GH], GH);
                }
                pg = seg_sum(pg, G, lane) * inv_denom;
                pu = seg_sum(pu, G, lane) * inv_denom;
                if (m == 0) {
                    kg0 = pg;
                    ku0 = pu;
                } else {
                    kg1 = pg;
                    ku1 = pu;
                }
                if (live && g == 0 && !(q == K && P.lora)) ll_put(S.llA + p, ex ? silu_f(pg) * pu : 0.f, ep);
            }
        }
        // LoRA of the shared expert on the CTAs holding its rows: wait for
        // z_g, z_u, finish a_s = silu(g + s B_g z_g) * (u + s B_u z_u), publish
        // it and this CTA's partial sums of z_d = A_d a_s
        if (P.lora && n_own > 0) {
            if (cw) {
                const float zr = lane < 2 * rank ? ll_wait(S.llZg + lane, ep, cx) : 0.f;
#pragma unroll
                for (int m = 0; m < LL_MAXA; ++m) {
                    const int pw = P.A0 + (warp + LL_NW * m) * R;
                    for (int s = 0; s < R; ++s) {
                        const int p = pw + s;
                        if (p < P.ps0 || p >= P.A1) continue;  // warp-uniform
                        const float pg = __shfl_sync(0xffffffffu, m == 0 ? kg0 : kg1, s * G);
                        const float pu = __shfl_sync(0xffffffffu, m == 0 ? ku0 : ku1, s * G);
                        const int o = p - P.ps0;
                        float dg = 0.f, du = 0.f;
                        if (lane < rank) dg = __half2float(gbg[(size_t)o * rank + lane]) * zr;
                        else if (lane < 2 * rank) du = __half2float(gbu[(size_t)o * rank + lane - rank]) * zr;
                        dg = warp_sum(dg);
                        du = warp_sum(du);
                        if (lane == 0) {
                            const float as = silu_f(fmaf(L.lscale, dg, pg)) * fmaf(L.lscale, du, pu);
                            ll_put(S.llA + p, as, ep);
                            aso[o] = as;
                        }
                    }
                }
            }
            __syncthreads();
            if (warp < rank) {
                const float v = warp_sum(lane < n_own ? h2f(adh) * aso[lane] : 0.f);
                if (lane == 0) ll_put(S.llZd + (size_t)(c - P.sh0) * LL_RANK + warp, v, ep);
            }
        }

        // ---- head work off the critical path: publish the previous layer's
        // head sums; this layer's fc1 / linear-residual rows (published in the
        // next layer)
        const int hidp = P.head_prev ? lyr[l - 1].hidden : 0;
        if (cw) {
            if (lp >= 0) combine(lp, h2f(b1h), h2f(b2h), zrp ? zdp[tid] : 0.f);
            if (P.head) {
#pragma unroll
                for (int m = 0; m < LL_MAXB1; ++m) {
                    const int it = warp + LL_NW * m;
                    if (it < nb1) {
                        const int ch = it % NC;
                        const uint4 wv = *reinterpret_cast<const uint4*>(
                            smem + lay.g_rows + ((size_t)(it / NC) * H + ch * 256 + lane * 8) * 2);
                        const float4 a0 = *reinterpret_cast<const float4*>(r + ch * 256 + lane * 8);
                        const float4 a1 = *reinterpret_cast<const float4*>(r + ch * 256 + lane * 8 + 4);
                        const float v = warp_sum(h8_dot44(wv, a0, a1));
                        if (lane == 0) pb1[(l & 1) * LL_MAXB1 * LL_NW + it] = v * inv_denom;
                    }
                }
                const float oh = warp_sum(h2f(ohh));
                if (warp < nq && lane == 0) poh[(l & 1) * LL_MAXROWS + warp] = oh;
            }

            // ---- 4. gather the a-words (quantised by warp, one half-group unit
            // each), the partial sums of z_d, and the hidden words of owner l-1's head.
            // Only a CTA with down rows reads the a-words and z_d sums: one without
            // rows publishes no residual word, so nothing keeps the other CTAs from
            // running a layer ahead and overwriting these words while it still reads them.
            const int nua = P.J1 > P.J0 ? P.NU : 0;
            unsigned long long aw[LL_MAXQ];
#pragma unroll
            for (int m = 0; m < LL_MAXQ; ++m) {
                const int u = warp + LL_NW * m;
                if (u < nua) aw[m] = ll_get(S.llA + u * 32 + lane);
            }
            const int nzd = P.lora && P.J1 > P.J0 ? P.nsh * rank : 0;
            unsigned long long zw = 0, hw = 0;
            const unsigned long long* zdw = S.llZd + (size_t)(tid / (rank > 0 ? rank : 1)) * LL_RANK +
                                            (rank > 0 ? tid % rank : 0);
            if (tid < nzd) zw = ll_get(zdw);
            const unsigned long long* hpw = S.llHp + (size_t)((l - 1) & 1) * (hidp + E);
            if (tid < hidp) hw = ll_get(hpw + tid);
#pragma unroll
            for (int m = 0; m < LL_MAXQ; ++m) {
                const int u = warp + LL_NW * m;
                if (u < nua) {
                    const float v = ll_take(aw[m], S.llA + u * 32 + lane, ep, cx);
                    quantize_half_warp(v, apl + u * 4, axg + u, lane);
                }
            }
            if (tid < nzd) zdp[tid] = ll_take(zw, zdw, ep, cx);
            for (int q = tid + LL_NW * 32; q < nzd; q += LL_NW * 32)
                zdp[q] = ll_wait(S.llZd + (size_t)(q / rank) * LL_RANK + q % rank, ep, cx);
            for (int q = tid; q < hidp; q += LL_NW * 32)
                ghp[q] = gelu_erf_f(q == tid ? ll_take(hw, hpw + q, ep - 1, cx) : ll_wait(hpw + q, ep - 1, cx));
        }
        if (__syncthreads_or(bad)) {
            leave();
            return;
        }
        // the gate/up buffer was last read above: the next layer's rows
        if (warp == PROD) {
            if (l + 1 < le && !layer_native(S, lyr[l + 1], t)) issue_g(l + 1);
        } else {
            if (P.lora && tid < rank) {
                float z = 0.f;
                for (int s = 0; s < P.nsh; ++s) z += zdp[s * rank + tid];
                zv[2 * LL_RANK + tid] = z;
            }

            // ---- 5. down: lane = output row (two half-warps), the warp's half-group
            // units; partial sums per (warp, half) summed across warps
            wait_bar(&bars[3], wt_d);
            const int half = lane >> 4, jr = lane & 15;
            float acc = 0.f;
            if (jr < NR) {
                for (int m = 0;; ++m) {
                    const int u = warp + LL_NW * (2 * m + half);
                    if (u >= P.NU) break;
                    const int q = u / HG, gi = (u % HG) >> 1;
                    if (!sl_l[q]) continue;
                    const uint4 cv = *reinterpret_cast<const uint4*>(dcodes + ((size_t)u * NRM + jr) * 16);
                    const uint32_t sv = *reinterpret_cast<const uint32_t*>(dsb + ((size_t)(q * GI + gi) * NRM + jr) * 4);
                    acc = fmaf(q < K ? wts[q] : 1.f, q4_half_dot(cv, apl + u * 4, axg[u], sv), acc);
                }
            }
            ypart[(warp * 2 + half) * LL_MAXROWS + jr] = acc;
        }
        __syncthreads();
        if (tid < NR) {
            const int j = P.J0 + tid;
            float y = 0.f;
            for (int p = 0; p < 2 * LL_NW; ++p) y += ypart[p * LL_MAXROWS + tid];
            if (P.lora) {
                const __half* bd = reinterpret_cast<const __half*>(hb + lay.h_bd) + (size_t)tid * rank;
                float d = 0.f;
                for (int rr = 0; rr < rank; ++rr) d = fmaf(__half2float(bd[rr]), zv[2 * LL_RANK + rr], d);
                y = fmaf(L.lscale, d, y);
            }
            const float rn = r[j] + y;
            ll_put(S.llR + j, rn, ep);
            if (l == Lz - 1) {
                r_out[j] = rn;
                if (tr.r) tr.r[(size_t)Lz * H + j] = rn;
            }
        }
        if (warp == PROD) {
            // the down buffer was last read above: the next layer's slices
            if (l + 1 < le && !layer_native(S, lyr[l + 1], t)) issue_d(l + 1);
        } else if (P.head_prev) {
            // ---- 6. fc2 rows of owner l-1 (published in the next layer)
            const int NCF = hidp / 256;
            const int nb2 = (P.F1 - P.F0) * NCF;
            if (warp < nb2) {
                const int ch = warp % NCF;
                const uint4 wv = *reinterpret_cast<const uint4*>(
                    hb + lay.h_f2 + ((size_t)(warp / NCF) * hidp + ch * 256 + lane * 8) * 2);
                const float4 a0 = *reinterpret_cast<const float4*>(ghp + ch * 256 + lane * 8);
                const float4 a1 = *reinterpret_cast<const float4*>(ghp + ch * 256 + lane * 8 + 4);
                const float v = warp_sum(h8_dot44(wv, a0, a1));
                if (lane == 0) pb2[(l & 1) * LL_NW + warp] = v;
            }
        }
        pend = l;
    }

    // ---- end of the launch: publish the last head sums, then route every head
    // whose logits were completed in this launch (owners lb-1 .. le-2) into the
    // prediction for the next token
    unsigned short b1h = 0, b2h = 0;
    float zrv = 0.f;
    if (pend >= 0 && cw) {
        combine_bias(pend, b1h, b2h);
        const unsigned long long* zrp = zres_word(pend);
        if (zrp) zrv = ll_wait(zrp, ep0 + pend - 1, cx);
    }
    if (__syncthreads_or(bad)) {
        leave();
        return;
    }
    if (pend >= 0 && cw) combine(pend, h2f(b1h), h2f(b2h), zrv);
    __syncthreads();
    for (int o = max(lb - 1, 0); o <= le - 2; ++o) {
        if (!lyr[o].fc1 || o % nb != c) continue;
        for (int e = tid; e < E; e += LL_THREADS) lg[e] = ll_wait(S.llZ + (size_t)o * E + e, ep0 + o + 1, cx);
        if (__syncthreads_or(bad)) {
            leave();
            return;
        }
        if (warp == 0) {
            const int np = (t + 1) & 1;
            int32_t* pi = S.pred_inds + ((size_t)np * Lz + (o + 1)) * K;
            float* pw = S.pred_w + ((size_t)np * Lz + (o + 1)) * K;
            RouteP rp = S.rp;
            rp.logit_bias = nullptr;
            route_warp_t<C::MAXM>(lg, E, rp, pi, pw, scr, st, lane);
            __syncwarp();
            if (tr.pred_inds && lane < K) tr.pred_inds[(size_t)(o + 1) * K + lane] = pi[lane];
        }
        __syncthreads();
    }
    leave();
    if (le == Lz && c == 0 && tid == 0) Sp->t = t + 1;
}
