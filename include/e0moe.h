/*
 * e0moe.h — C ABI of the GB300 (sm_103a) int4 gathered-expert MoE block, the
 * decode/prefill hot path of the Edge0 streaming-MoE engine.
 *
 * Sources, cited by page title and section:
 *   [KOALA]  "Edge0: 35B MoE를 SSD에서 3GiB 메모리로 서빙하기 — 라우팅을 한 토큰
 *            먼저 예측한다" (koala.ai.kr).
 *   [PTKR]   "edge0: 35B MoE 모델을 활성 메모리 3GiB로 실행하는 SSD 전문가
 *            스트리밍 추론 프레임워크" (discuss.pytorch.kr).
 *   [JAEHUN] "The Other Half of the Memory Wall: Serving 35B MoEs from SSD with
 *            Trained Routing Prediction" (jaehun.me review; cites paper sections).
 *   [XYZNOT] same title (xyznot.com summary).
 *
 * Conventions for every entry point
 *   - Pointers named d_* or documented "device" are device pointers owned by
 *     the caller; the library never frees or keeps them.  Pointers documented
 *     "host" are read during the call only.
 *   - fp16 data is passed as uint16_t (IEEE binary16 bits).
 *   - Calls are asynchronous on the given stream (a cudaStream_t; NULL = the
 *     legacy default stream) and never synchronise the host, except
 *     e0_read_status, e0_stack_prepare and e0_pack_experts where stated.
 *   - No call allocates memory.  Scratch comes from a caller workspace whose
 *     size the matching *_workspace_size function reports; it needs 256-byte
 *     alignment and its contents are not preserved across calls unless stated.
 *   - Return value: E0_OK or a negative E0_ERR_* code.  Arguments are checked
 *     on the host before anything is launched; a call that fails its checks
 *     launches nothing.
 *   - Conditions found on the device (a routed expert with no slot, an expert
 *     id out of range, a non-finite logit, an exhausted wait) never trap: they
 *     OR E0_ST_* bits into the caller's d_status word (when non-NULL) and the
 *     affected contribution is zero.  e0_read_status copies the word back.
 *
 * Canonical int4 projection ("Q-tensor") for a matrix with `out` rows and `in`
 * inputs — affine int4 with group size 64 along the input dimension ([KOALA]
 * §1 "SSD 스트리밍 전문가 레이어" and the tier table "두 공개 티어"; [PTKR]
 * "SSD 전문가 스트리밍"):
 *     codes  uint8  [out][in/2]   element j of a row: byte j/2, low nibble when
 *                                 j is even, high nibble when j is odd (q 0..15)
 *     scale  fp16   [out][in/64]
 *     bias   fp16   [out][in/64]
 *     w[o][j] = scale[o][j/64] * q[o][j] + bias[o][j/64]
 * An expert is gate [I][H], up [I][H], down [H][I]; y = down(silu(gate x) *
 * up x) ([JAEHUN] "새로운 접근법: Edge0", paper §3.1 math contract).
 *
 * Kernel ("slot") layout of one expert, produced by e0_pack_experts, in
 * e0_slot_bytes(H, I) bytes:
 *     [0, I*H)                 gate/up codes, row-interleaved: for each i the
 *                              gate row i (H/2 bytes) then the up row i
 *     [I*H, I*H + H*I/2)       down codes in blocks of 16 output rows: the
 *                              16 bytes of row j, inputs 32c..32c+31, at
 *                              ((j/16 * I/32 + c) * 16 + j%16) * 16
 *     next I*(H/64)*2*4 bytes  gate/up (scale, bias) fp16 pairs, [I][2][H/64]
 *     next H*(I/64)*4 bytes    down (scale, bias) fp16 pairs in the same
 *                              row blocks: group g of row j at
 *                              ((j/16 * I/64 + g) * 16 + j%16) * 4
 * (Every input of a block of 16 output rows is one contiguous range of codes
 * and one of (scale, bias) words, so a decode block's share of the down
 * projection is two bulk copies per expert.)  Inside every 32-bit word (8
 * elements e0..e7 of a row) the nibbles are interleaved: nibble j (bits
 * 4j..4j+3, little-endian word) holds e0, e2, e4, e6, e1, e3, e5, e7 for
 * j = 0..7.  Masking a word with 0x000F000F / 0x00F000F0 (and the same after
 * a shift by 8) then yields consecutive element pairs, and masking with
 * 0x0F0F0F0F yields four byte lanes.  H and I must be multiples of 64 and at
 * most 2048.
 */
#ifndef E0MOE_H
#define E0MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* e0_stream_t; /* the same handle as cudaStream_t */

/* ---- return codes ---------------------------------------------------- */
enum {
    E0_OK = 0,
    E0_ERR_ARG = -1,         /* a shape, size or option is invalid          */
    E0_ERR_NULL = -2,        /* a required pointer is NULL                  */
    E0_ERR_UNSUPPORTED = -3, /* valid but outside what the kernels support  */
    E0_ERR_CUDA = -4         /* a CUDA launch or copy returned an error     */
};

/* ---- device status bits (OR-ed into *d_status) ------------------------ */
enum {
    E0_ST_SLOT_MISS = 1u,    /* a routed expert has no slot: contributes 0  */
    E0_ST_BAD_EXPERT = 2u,   /* an expert id outside [0, E): ignored        */
    E0_ST_NONFINITE = 4u,    /* a routing score was NaN or infinite         */
    E0_ST_TIMEOUT = 8u,      /* a bounded device-side wait gave up          */
    E0_ST_POOL_FULL = 16u,   /* slot_update found no free slot              */
    E0_ST_INTERNAL = 32u     /* a kernel's own consistency check failed; the
                                step was skipped (results are not valid)    */
};

/* ---- routing rules -------------------------------------------------- */
enum { E0_ROUTE_SOFTMAX_TOPK = 0, E0_ROUTE_SIGMOID_GROUP = 1 };

/* Limits of the kernels (E0_ERR_UNSUPPORTED beyond them). */
enum { E0_MAX_E = 1024, E0_MAX_K = 32, E0_MAX_T_DECODE = 64, E0_MAX_LORA_RANK = 64 };

typedef struct e0_qtensor {
    const uint8_t* codes;    /* device, [out][in/2]  */
    const uint16_t* scale;   /* device, fp16 [out][in/64] */
    const uint16_t* bias;    /* device, fp16 [out][in/64] */
} e0_qtensor;

typedef struct e0_expert_q {
    e0_qtensor gate, up, down;
} e0_expert_q;

/* A slot pool: n_slots experts in the kernel layout plus the slot table that
 * maps an expert id to its slot ([KOALA] §1 staged path; [JAEHUN] paper §3.1:
 * routing indices reach the slots through a table, so they never leave the
 * GPU).  A resident bank is a pool with n_slots == E and the identity table. */
typedef struct e0_slot_pool {
    uint8_t* data;           /* device, n_slots * e0_slot_bytes(H, I) bytes  */
    int32_t* slot_table;     /* device [E]: expert -> slot, -1 = absent      */
    int32_t* occupant;       /* device [n_slots]: slot -> expert, -1 = empty */
    int32_t n_slots, H, I, E;
} e0_slot_pool;

typedef struct e0_route_params {
    int32_t mode;            /* E0_ROUTE_SOFTMAX_TOPK or E0_ROUTE_SIGMOID_GROUP */
    int32_t K;               /* experts per token, 1 <= K <= min(E, 32)         */
    int32_t n_groups;        /* sigmoid-group: n, E % n == 0                    */
    int32_t topk_groups;     /* sigmoid-group: G, 1 <= G <= n                   */
    float scale;             /* sigmoid-group: s                                */
    const float* logit_bias; /* device [E] added to router logits, or NULL      */
} e0_route_params;

/* Shared expert: one expert in the kernel layout plus an optional unmerged
 * LoRA on each projection, P(x) = W_int4 x + (alpha/rank) B (A x)
 * ([XYZNOT] "Ausführung des unzusammengeführten Adapters"; [KOALA] §3).
 * A_* fp16 [rank][in], B_* fp16 [out][rank]; all six NULL = no LoRA. */
typedef struct e0_shared_expert {
    const uint8_t* data;     /* device, e0_slot_bytes(H, I) bytes, kernel layout */
    const uint16_t* A_gate; const uint16_t* B_gate;
    const uint16_t* A_up;   const uint16_t* B_up;
    const uint16_t* A_down; const uint16_t* B_down;
    int32_t rank;
    float alpha;
} e0_shared_expert;

/* Prerouter head owned by layer N, predicting layer N+1 at token t+1
 * ([XYZNOT] "Architektur des Prerouter-Heads": head(f) = fc2(gelu_erf(fc1 f))
 * + l(f), f = [h ; onehot(top-K now) ; onehot(top-K previous token)],
 * dim = H + 2E).  fp16 weights: fc1 [hidden][H+2E], b1 [hidden] or NULL,
 * fc2 [E][hidden], b2 [E] or NULL, lres [E][H+2E] (the linear residual). */
typedef struct e0_prerouter {
    const uint16_t* fc1; const uint16_t* b1;
    const uint16_t* fc2; const uint16_t* b2;
    const uint16_t* lres;
    int32_t H, E, hidden;
} e0_prerouter;

/* ---- sizes ------------------------------------------------------------ */

/* Bytes of one expert in the kernel layout (equal to the canonical size). */
size_t e0_slot_bytes(int H, int I);

/* Workspace for e0_moe_block_forward / e0_prerouter_forward /
 * e0_moe_prefill_forward.  op: 0 = moe_block_forward, 1 = prerouter_forward,
 * 2 = moe_prefill_forward.  For op 1, I is read as the head's hidden width. */
size_t e0_workspace_size(int op, int T, int H, int I, int E, int K);

/* ---- packing and the slot table --------------------------------------- */

/* Convert n experts from the canonical layout into pool slots: src[i] (host
 * array of device descriptors) goes to slot dst_slots[i] (host array).  When
 * expert_ids (host [n]) is non-NULL, also sets slot_table[expert_ids[i]] =
 * dst_slots[i] and occupant[dst_slots[i]] = expert_ids[i] on the device.
 * Not a hot-path call: it launches one kernel per expert and synchronises the
 * stream before returning (the host arrays may be freed afterwards). */
int e0_pack_experts(const e0_expert_q* src, int n, const e0_slot_pool* dst,
                    const int32_t* dst_slots, const int32_t* expert_ids, e0_stream_t stream);

/* Incremental in-place slot update (incr_stack: [KOALA] §1 staged path and
 * 한계; [JAEHUN] paper §3.1 and Appx.B; [XYZNOT] "incremental sticky-slot
 * stack").  For the next set d_inds_next [n_next] (device), copies every
 * expert that has no slot from `bank` (device or host-mapped memory holding
 * all E experts in the kernel layout, expert e at bank + e*e0_slot_bytes) into
 * the lowest-numbered free slot, then updates slot_table and occupant.  A slot
 * is free when it holds no expert of d_inds_cur [n_cur] (may be NULL) nor of
 * the next set.  Only changed slots are written; a resident bank (every
 * expert already has a slot) moves zero bytes.  No free slot left: sets
 * E0_ST_POOL_FULL and leaves that expert absent.  Ids outside [0, E) set
 * E0_ST_BAD_EXPERT and are skipped.  One block plans the copies (each block
 * replays the plan); the bytes move with 16-byte copies spread over one
 * block per SM, then one block commits the tables. */
int e0_slot_update(const e0_slot_pool* pool, const int32_t* d_inds_next, int n_next,
                   const int32_t* d_inds_cur, int n_cur, const uint8_t* bank,
                   uint32_t* d_status, e0_stream_t stream);

/* ---- routing (softmax-top-k and sigmoid group-limited top-k) ---------- */

/* Softmax-top-k ([JAEHUN] "새로운 접근법: Edge0", paper Appx.A):
 * g = softmax(l); inds = top-k(g, K); w = g[inds] / sum(g[inds]).
 * logits fp32 [T][E] device; inds int32 [T][K] (descending score, ties to the
 * lower expert id); w fp32 [T][K].  One warp per token. */
int e0_route_softmax_topk(const float* logits, int T, int E, int K, int32_t* inds, float* w,
                          uint32_t* d_status, e0_stream_t stream);

/* Sigmoid group-limited top-k (same passage): sigma = sigmoid(l); groups are
 * n contiguous blocks of E/n experts; a group's score is the sum of its two
 * largest sigma; the best G groups are kept (ties to the lower group); inds =
 * top-k(sigma, K) over kept groups; w = s*sigma[inds]/(sum sigma[inds] + 1e-20).
 * Requires K <= G*E/n. */
int e0_route_sigmoid_group(const float* logits, int T, int E, int n_groups, int topk_groups,
                           int K, float s, int32_t* inds, float* w, uint32_t* d_status,
                           e0_stream_t stream);

/* h = r / sqrt(mean(r^2) + eps), no learned weight (the post-attention norm
 * whose output feeds the MoE block and the head; [KOALA] §2).  fp32 [T][H]. */
int e0_rmsnorm(const float* r, int T, int H, float eps, float* h, e0_stream_t stream);

/* ---- decode MoE block ------------------------------------------------- */

/* y = sum_k w_k * expert_{inds_k}(x) (+ shared(x)) for T decode tokens
 * ([JAEHUN] paper §3.1 math contract and Appx.A; [KOALA] §2 prediction as
 * routing).  x fp32 [T][H] device (the MoE input h).  Experts are read in
 * place from `pool` through its slot table.
 * Routing: when inds_in is NULL the block routes natively: logits = W_router
 * x (+ rp->logit_bias), W_router fp16 [E][H], then rp's rule.  When inds_in
 * (int32 [T][K]) and w_in (fp32 [T][K]) are given, that routing is used as is
 * (a prediction made one token earlier); W_router may then be NULL.
 * inds_out / w_out (may be NULL) receive the routing used.  shared may be
 * NULL.  Output y fp32 [T][H].  T <= 64. */
int e0_moe_block_forward(const float* x, int T, const e0_slot_pool* pool,
                         const uint16_t* W_router, const e0_route_params* rp,
                         const int32_t* inds_in, const float* w_in,
                         const e0_shared_expert* shared,
                         float* y, int32_t* inds_out, float* w_out,
                         void* ws, size_t ws_bytes, uint32_t* d_status, e0_stream_t stream);

/* Same computation as e0_moe_block_forward, for callers that cannot hand the
 * library a workspace: a plugin inside a host framework that owns every device
 * allocation, or a serving loop with a fixed memory plan that must not
 * allocate once it runs.  There is no counterpart on the pages this library
 * follows; it is a deployment convenience.  The scratch is a fixed device
 * array of E0_NOALLOC_SCRATCH_BYTES inside the library (each GPU that loads
 * the library holds it until the process exits); a call whose workspace need
 * (e0_workspace_size(0, ...)) exceeds it returns E0_ERR_UNSUPPORTED and
 * launches nothing.  The call allocates nothing.  The first call on a device
 * looks up the array's device address with that device current; make that
 * first call before any stream capture.  All calls share the one array and it
 * keeps the previous call's contents (nothing in it needs to start at zero):
 * calls whose work overlaps on the GPU (other streams, other threads) race on
 * it, so serialise them. */
#define E0_NOALLOC_SCRATCH_BYTES (1u << 20)
int e0_moe_block_forward_noalloc(const float* x, int T, const e0_slot_pool* pool,
                                 const uint16_t* W_router, const e0_route_params* rp,
                                 const int32_t* inds_in, const float* w_in,
                                 const e0_shared_expert* shared,
                                 float* y, int32_t* inds_out, float* w_out,
                                 uint32_t* d_status, e0_stream_t stream);

/* Prerouter head for T tokens: z = fc2 gelu_erf(fc1 f + b1) + b2 + lres f with
 * f = [h ; onehot(inds_cur) ; onehot(inds_prev)] (inds_prev NULL = all zeros,
 * the first token), then rp's routing of z gives the next layer's routing for
 * the next token ([PTKR] "라우팅을 한 스텝 먼저 예측하는 프리라우터"; [JAEHUN]
 * "작동 원리" toy example).  h fp32 [T][H]; inds_cur/inds_prev int32 [T][K];
 * logits_out fp32 [T][E] (may be NULL); inds_next [T][K]; w_next [T][K]. */
int e0_prerouter_forward(const float* h, int T, const int32_t* inds_cur, const int32_t* inds_prev,
                         const e0_prerouter* head, const e0_route_params* rp,
                         float* logits_out, int32_t* inds_next, float* w_next,
                         void* ws, size_t ws_bytes, uint32_t* d_status, e0_stream_t stream);

/* ---- decode stack (one token through L layers) ----------------------- */

/* One layer of a decode stack.  `pool` holds the layer's experts (normally
 * the resident bank); W_router fp16 [E][H] routes the layer natively (every
 * layer at the first token, non-consumers always); `consumer` = 1 makes the
 * layer route with the prediction its owner made one token earlier once one
 * exists; `head` (or NULL) is the prerouter this layer owns; `shared` may be
 * NULL.  The descriptors pointed to are copied by e0_stack_prepare. */
typedef struct e0_stack_layer {
    e0_slot_pool pool;
    const uint16_t* W_router;
    const e0_shared_expert* shared;
    const e0_prerouter* head;
    int32_t consumer;
} e0_stack_layer;

/* Optional per-token trace (device buffers; any may be NULL):
 * r [L+1][H] residual stream at every layer input and the output,
 * inds/w [L][K] the routing each layer used, head_logits [L][E] the logits of
 * the head each owner evaluated (rows of non-owners untouched),
 * pred_inds [L][K] the routing predicted for each consumer for the next token. */
typedef struct e0_stack_trace {
    float* r;
    int32_t* inds;
    float* w;
    float* head_logits;
    int32_t* pred_inds;
} e0_stack_trace;

/* Workspace of a stack (state carried between tokens lives here). */
size_t e0_stack_workspace_size(int L, int H, int I, int E, int K, int head_hidden);

/* Copy the layer descriptors into the workspace and clear the routing
 * history and the flag-carrying words (the next step is token 0).
 * Synchronises the stream.  Also sizes the flag-carrying-word kernel (impl 3):
 * one block of 17 warps per SM and the shared memory that stages each
 * layer's weight slices.  Environment (read here): E0MOE_WAIT_US (1..10^7,
 * default 200000) is the longest a device-side wait of impl 3 polls before
 * it gives up with E0_ST_TIMEOUT; E0MOE_PF_DIST (0..64, default 0) makes
 * impl 3 also prefetch the weights of that many layers ahead into L2;
 * E0MOE_LL_FREE_SMS (0..64, default 0) launches impl 3 on that many fewer
 * SMs, so that kernels on other streams (host-tier slot copies) can run
 * beside it (a stack whose work split no longer fits then gets
 * E0_ERR_UNSUPPORTED from impl 3). */
int e0_stack_prepare(const e0_stack_layer* layers, int L, int H, int I, int E,
                     const e0_route_params* rp, void* ws, size_t ws_bytes, e0_stream_t stream);

/* Decode one token: r_0 = x; for each layer h = rmsnorm(r) (eps 1e-6);
 * route (prediction or native); r += MoE(h) + Shared(h); owners evaluate their
 * head and store the next token's routing for layer+1.  x fp32 [H] device,
 * r_out fp32 [H] device.  impl selects the kernels (same arithmetic):
 *   0 = one persistent cooperative kernel per token, two or three grid
 *       barriers per layer (deterministic);
 *   1 = a chain of per-phase kernels (deterministic, equal to 0 bit for bit);
 *   2 = retired: returns E0_ERR_UNSUPPORTED;
 *   3 = one cooperative launch per token of the flag-carrying-word kernel:
 *       blocks exchange the layer's activations and residual rows through
 *       64-bit (epoch, value) words instead of grid barriers, and stage every
 *       weight slice with bulk copies issued a layer ahead where the routing
 *       is known (deterministic; sums in another order than 0).  Built for
 *       the layer shapes (H, I, E, K) = (2048, 512, 256, 2 / 4 / 8),
 *       (1536, 384, 128, 8), (256, 128, 16, 4) with LoRA ranks 8 or 16;
 *       other stacks -> E0_ERR_UNSUPPORTED (use 0).  A device-side wait that
 *       gives up sets E0_ST_TIMEOUT in d_status and a flag in the workspace
 *       that makes every later impl-3 step of it give up at once: prepare
 *       the stack again after a timeout. */
int e0_stack_step(const float* x, float* r_out, void* ws, const e0_stack_trace* trace,
                  int impl, uint32_t* d_status, e0_stream_t stream);

/* ---- staged streaming of predicted experts ------------------------------ */

/* Layers [layer_begin, layer_end) of the current token with the
 * flag-carrying-word kernel (impl 3).  A token is the launches whose ranges cover 0..L in order
 * on one stream; x is read by the range that starts at 0, r_out written by
 * the range that ends at L (the token counter advances there).  Between the
 * launches of a token the caller may run other work on other streams, e.g.
 * e0_stack_prefetch_experts for layers whose prediction for the next token
 * is already final.  ([KOALA] §1-§2, [JAEHUN] §3.1: the prediction made one
 * token ahead is what lets the load of the next token's experts overlap the
 * current token.)  Errors: unknown workspace or empty / out-of-range layer
 * range -> E0_ERR_ARG; a stack impl 3 is not built for -> E0_ERR_UNSUPPORTED. */
int e0_stack_step_range(const float* x, float* r_out, void* ws, int layer_begin, int layer_end,
                        const e0_stack_trace* trace, uint32_t* d_status, e0_stream_t stream);

/* Replace the layer descriptors of a prepared stack (e.g. move a layer from
 * the resident bank to a staged slot pool) keeping its routing history,
 * predictions and token counter.  Each layer must keep its configuration
 * (shared expert, LoRA rank, head, consumer flag) -> else E0_ERR_ARG.
 * Synchronises the stream. */
int e0_stack_update_layers(void* ws, const e0_stack_layer* layers, int L, e0_stream_t stream);

/* Bring the K experts the prerouter predicted for token t_next (>= 1) of
 * `layer` into `pool` (a staged slot pool whose table the layer's descriptor
 * uses): e0_slot_update from `bank` (the layer's experts in kernel layout,
 * device or host memory the GPU can read, slot i = expert i) with the
 * prediction as the next set.  Valid once the prediction is final: after the
 * launch that ran layer + 1 of token t_next - 1 (or that token's last layer). */
int e0_stack_prefetch_experts(void* ws, int layer, int t_next, const e0_slot_pool* pool, const uint8_t* bank,
                              uint32_t* d_status, e0_stream_t stream);

/* e0_stack_prefetch_experts for n layers at once: layers[i] into pools[i]
 * from banks[i] (host arrays of n entries, 0 <= n <= 64, every pool of one H
 * and I, no pool twice).  One copy launch covers every layer's missing
 * experts and one commit launch updates every table, instead of two launches
 * a layer; the result is that of n calls of e0_stack_prefetch_experts.
 * Errors: a NULL array or bank -> E0_ERR_NULL; n out of range, a layer out of
 * range, pools of different H / I or a pool given twice -> E0_ERR_ARG; a
 * pool failing e0_slot_update's checks -> its code. */
int e0_stack_prefetch_experts_batch(void* ws, const int32_t* layers, int n, int t_next,
                                    const e0_slot_pool* pools, const uint8_t* const* banks,
                                    uint32_t* d_status, e0_stream_t stream);

/* A cross-layer cache of expert bundles in device memory, least recently used
 * first out ([PTKR] "SSD 전문가 스트리밍" / P2 `SharedExpertCache`: a hot set
 * shared by all layers; misses go to the exact path, here the host bank).
 * Keys are layer * E + expert.  All arrays are device memory owned by the
 * caller and start as: key = -1, stamp = 0, map = -1, counters = 0. */
typedef struct e0_expert_cache {
    uint8_t* data;        /* capacity * e0_slot_bytes(H, I) bytes              */
    int32_t* key;         /* [capacity] key held by each entry, -1 = empty      */
    uint32_t* stamp;      /* [capacity] last use (a counter), 0 = never         */
    int32_t* map;         /* [n_keys] key -> entry, -1 = not cached             */
    uint32_t* counters;   /* [4]: clock, hits, misses, evictions                */
    int32_t* scratch;     /* [4 + 4 * E0_MAX_K] plan of one prefetch           */
    int32_t capacity, n_keys;
} e0_expert_cache;

/* e0_stack_prefetch_experts with a cross-layer cache in front of `bank`: a
 * predicted expert missing from the layer's pool is copied from its cache
 * entry when it has one (device to device), else from `bank` — and then also
 * into the least recently used cache entry not used by this call (with none
 * left, the expert is not cached).  Hits, misses and evictions are
 * counted in cache->counters.  Errors as e0_stack_prefetch_experts; a layer
 * * E key beyond n_keys -> E0_ERR_ARG. */
int e0_stack_prefetch_experts_cached(void* ws, int layer, int t_next, const e0_slot_pool* pool,
                                     const uint8_t* bank, const e0_expert_cache* cache,
                                     uint32_t* d_status, e0_stream_t stream);

/* e0_stack_prefetch_experts_cached for n layers at once, with the arrays and
 * limits of e0_stack_prefetch_experts_batch: one launch plans every layer in
 * order (the cache's recency order is that of n calls in the order given),
 * one copies, one commits.  An entry used by one layer of the batch (as a
 * source or filled) is not evicted for another layer of the same batch; with
 * every entry so taken, an expert is copied from its bank without being
 * cached.  The plans live in the stack workspace (cache->scratch is not used).
 * Errors as e0_stack_prefetch_experts_batch and
 * e0_stack_prefetch_experts_cached. */
int e0_stack_prefetch_experts_cached_batch(void* ws, const int32_t* layers, int n, int t_next,
                                           const e0_slot_pool* pools, const uint8_t* const* banks,
                                           const e0_expert_cache* cache, uint32_t* d_status,
                                           e0_stream_t stream);

/* ---- whole-layer prefill (sorted gather + tcgen05 grouped GEMM) ------- */

/* Group the T*K assignments (t, k) by expert ([PTKR] "SSD 전문가 스트리밍":
 * the full-layer path computes with a sorted gather).  counts [E], offsets
 * [E+1] (exclusive scan), perm [T*K]: assignment ids t*K+k ordered by expert,
 * token order kept within an expert. */
int e0_prefill_sort(const int32_t* inds, int T, int K, int E, int32_t* counts, int32_t* offsets,
                    int32_t* perm, void* ws, size_t ws_bytes, e0_stream_t stream);

/* Prefill one layer for T tokens: route every token natively (logits =
 * W_router X + rp->logit_bias, on the tensor cores with fp32 accumulation; a
 * token whose K+1 largest scores, or whose G-th and (G+1)-th group scores,
 * lie closer than 2e-4 is routed again from fp32 SIMT dot products, the
 * precision of the decode path), sort assignments by expert, gather X rows,
 * run gate/up and down as grouped GEMMs on the tensor cores (fp16 operands,
 * weights dequantised on chip, fp32 accumulation), and form Y[t] =
 * sum_k w[t][k] expert(X[t]): added in fp32 with atomics (the order of the K
 * terms varies between runs), or, with the environment variable
 * E0MOE_PREFILL_FIXED_ORDER=1 at the call, summed from fp16 rows in a fixed
 * order (the same bits on every run).  X fp16 [T][H]; bank = the
 * layer's experts (slot table consulted per expert); Y fp32 [T][H];
 * inds_out/w_out [T][K].  Prefill never predicts ([JAEHUN] "작동 원리"). */
int e0_moe_prefill_forward(const uint16_t* X, int T, const e0_slot_pool* bank,
                           const uint16_t* W_router, const e0_route_params* rp,
                           float* Y, int32_t* inds_out, float* w_out,
                           void* ws, size_t ws_bytes, uint32_t* d_status, e0_stream_t stream);

/* ---- status ------------------------------------------------------------- */

/* Largest wait e0_selftest_bounded_wait accepts, in microseconds. */
#define E0_SELFTEST_MAX_WAIT_US 2000000u

/* Exercise the device-side bounded wait that guards every spin in this
 * library (grid barriers of the stack kernels, pipeline barriers of the
 * prefill GEMMs): one thread polls *flag (caller-owned device word) until it
 * is non-zero or limit_us microseconds of device time (globaltimer) have
 * passed; on the time limit it ORs E0_ST_TIMEOUT into *d_status and returns.
 * Nothing traps, so the context stays usable and a later e0_read_status
 * reports the bit.  The pages describe no such call: it lets a caller (and the
 * tests) check that a wait which never ends is turned into a status bit.
 * Errors: NULL flag or d_status -> E0_ERR_NULL; limit_us == 0 or above
 * E0_SELFTEST_MAX_WAIT_US -> E0_ERR_ARG. */
int e0_selftest_bounded_wait(const uint32_t* flag, uint32_t limit_us, uint32_t* d_status, e0_stream_t stream);

/* Copy *d_status to *h_out after everything queued on `stream`; synchronises
 * the stream. */
int e0_read_status(const uint32_t* d_status, uint32_t* h_out, e0_stream_t stream);

/* A static string describing a return code. */
const char* e0_status_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* E0MOE_H */
