/*
 * moe.h — C ABI of libmoe: the routed-expert MoE FFN layer at decode and
 * small-batch time (and its prefill grouped-GEMM path) on one GB300 (sm_103a).
 *
 * The layer: a router GEMV, top-k expert selection with a softmax over the
 * selected experts, block-quantised gate/up/down matvecs over the selected
 * experts only, SwiGLU, and a router-weighted combine.  Expert weights are
 * served from slot pools in device memory, one pool per type/shape group of
 * layers, managed least-recently-used, with misses uploaded from pinned host
 * memory on a side stream.
 *
 * Sources for the operations (web pages on llama.cpp MoE expert handling):
 *  - page 1, "llama.cpp MoE 模型卸载" blog, section 3.1 (gating: logits,
 *    softmax, partial_sort top-k), 3.2 (load on demand, LRU of non-active
 *    experts), 3.3 (device-side expert pointers for the FFN kernel);
 *  - page 2, "llama.cpp MoE GGUF 张量加载" notes (ffn_{gate,up,down}_exps
 *    expert-major tensors);
 *  - page 3, tiered MoE scheduling note (routed vs always-resident shared
 *    experts, pinned memory and async H2D copies);
 *  - page 4, "llama.cpp MoE缓存实测" (slot pools grouped by tensor type and
 *    shape, LRU shared across a group's layers, PCIe upload on miss, the
 *    <=32-token batch limit, the slot budget and its floor, hit statistics);
 *  - page 5, "GPU 卸载研究笔记" section 1.2 (quantised blocks kept as-is and
 *    multiplied by an on-GPU quantised GEMV).
 *
 * Conventions for every entry point:
 *  - Return value: a moe_status code (0 = MOE_OK).  Nothing aborts the process.
 *  - Pointers named d_* / "device" are device addresses; "host" pointers are
 *    host addresses.  Every buffer is owned by the caller; the library never
 *    frees caller memory and never allocates device memory the caller sees
 *    (library-owned objects — moe_cache, moe_stack — hold only host memory and
 *    CUDA events).
 *  - Calls taking a stream are asynchronous on that stream unless noted;
 *    argument errors are detected on the host before anything is enqueued.
 *  - Device-side faults that can only be seen on the GPU (an expert id or a
 *    slot out of range, a bounded wait that ran out) are recorded in a
 *    per-device status word read by moe_device_status(); the offending work is
 *    skipped, never trapped.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *moe_stream_t; /* the same type as cudaStream_t */

/* ------------------------------------------------------------------ status */

enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID = -1,     /* bad argument (null, shape, range, alignment, not pinned) */
    MOE_ERR_CUDA = -2,        /* a CUDA runtime call failed */
    MOE_ERR_CAPACITY = -3,    /* more distinct experts requested than the pool has slots */
    MOE_ERR_BUDGET = -4,      /* a pool too small for one request (page 4's budget floor) */
    MOE_ERR_TIMEOUT = -5,     /* a bounded device-side wait ran out */
    MOE_ERR_UNSUPPORTED = -6  /* a shape/type combination this build has no kernel for */
};

/* Static message for a status code; never NULL. */
const char *moe_status_string(int status);

/* Name of the CUDA error behind the calling thread's last MOE_ERR_CUDA ("none" if none). */
const char *moe_last_cuda_error(void);

/* Library limits. */
#define MOE_MAX_K 8          /* top-k limit (k <= 8 covers every workload) */
#define MOE_MAX_E 256        /* experts per layer */
#define MOE_DECODE_MAX_T 32  /* page 4: the slot cache serves batches of <= 32 tokens */

/* Quantisation formats of expert weights (canonical block layouts). */
enum moe_qtype {
    MOE_Q8_0 = 0,  /* 34 B per 32 weights: fp16 d (little-endian), int8 q[32]; w = d*q */
    MOE_Q4_SM = 1  /* 20 B per 32 weights: fp16 d, fp16 m, 16 B codes (byte i: q[2i] low
                      nibble, q[2i+1] high nibble); w = d*q + m */
};
/* Activation element types. */
enum moe_xtype { MOE_F32 = 0, MOE_BF16 = 1 };

/* --------------------------------------------------------------- router (a1, a2) */

/*
 * moe_router_topk — gating for T tokens (page 1, section 3.1).
 *   logits[t][e] = sum_h x[t][h] * w_router[h][e] + bias[e]   (fp32 accumulation)
 *   ids[t][:]     = the k experts with the largest logits, in descending logit order,
 *                   equal logits ordered by ascending expert id
 *   weights[t][j] = exp(l_j - l_max) / sum_{i in top-k} exp(l_i - l_max)
 * x        device [T][H], fp32 (xtype MOE_F32) or bf16 (MOE_BF16), row-major.
 * w_router device [H][E] fp16 bit patterns, row-major (E contiguous).
 * bias     device [E] fp32 or NULL.
 * ids      device [T][k] int32 out;  weights device [T][k] fp32 out.
 * logits   device [T][E] fp32 out, or NULL.
 * Limits: 1 <= k <= min(E, MOE_MAX_K), E <= MOE_MAX_E, H % 32 == 0, T >= 0 (T == 0: no-op).
 * Path: T <= MOE_DECODE_MAX_T one 8-CTA cluster per 32 tokens (fp32 FMAs); larger T with bf16
 * x, E a multiple of 32 up to 128 and H a multiple of 64 on tensor cores (bf16 values in the
 * normal fp16 range are exact in fp16, W_r is fp16: exact products, fp32 sums per 64 rows of
 * H); otherwise a tiled fp32 kernel.
 */
int moe_router_topk(const void *x, int xtype, int T, int H, const uint16_t *w_router,
                    const float *bias, int E, int k, int32_t *ids, float *weights,
                    float *logits, moe_stream_t s);

/*
 * moe_router_topk_threshold — moe_router_topk with the load threshold of page 1 (section
 * 4.3, --moe-expert-load-threshold 0.05: a selected expert whose gate score is below the
 * threshold is not loaded).  Reading: a route (t, j) whose weight (the softmax over the k
 * selected logits) is below min_weight is dropped: ids[t][j] = -1 and weights[t][j] = 0;
 * the other routes keep their weights (no renormalisation), so the layer's output loses
 * those terms (this variant changes the result).  Every other entry point treats id -1 as
 * "no route": it is skipped, not an error; moe_expert_ffn leaves partial[t][j] of such a
 * route untouched (the stack's combine skips it).  min_weight in [0, 1]; 0 drops nothing.
 */
int moe_router_topk_threshold(const void *x, int xtype, int T, int H, const uint16_t *w_router,
                              const float *bias, int E, int k, float min_weight, int32_t *ids,
                              float *weights, float *logits, moe_stream_t s);

/* ------------------------------------------------------------------ slot images */

/*
 * moe_slot_image_bytes — size of one expert's slot image (gate + up + down).
 * It equals the canonical size: 2*F*H/32*B + H*F/32*B with B = 34 (q8_0) or 20 (4-bit).
 * H and F must be multiples of 32.
 */
int moe_slot_image_bytes(int qtype, int H, int F, size_t *bytes_out);

/*
 * moe_pack_expert — host: canonical expert tensors -> one slot image.
 * gate_aos, up_aos: host [F rows][H/32 blocks] canonical blocks; down_aos: [H][F/32].
 * slot_image_dst: host buffer of moe_slot_image_bytes() bytes (16-byte aligned);
 * pass NULL to query the size only.  Layout of the image: gate [F][H], up [F][H], down
 * [H][F], each matrix a run of 32-row tiles, each tile a run of "tile blocks" (one per
 * 32-column block along K): first the codes of the 32 rows (q8_0: two 512-byte pieces,
 * row l's 16 codes of piece p at 512 p + 16 ((l + 4 p) mod 32), each stored as q + 128,
 * offset binary;
 * 4-bit: one 512-byte piece, row l's 16 canonical code bytes at 16 l), then the 32 rows'
 * scale entries (fp16 d, or fp16 d and m), row l's entry at position 4 (l % 8) + l / 8.
 * So any K range of a tile is one contiguous run of bytes.  The image has the canonical
 * size and holds the same values; moe_unpack_expert inverts it exactly.
 */
int moe_pack_expert(int qtype, int H, int F, const void *gate_aos, const void *up_aos,
                    const void *down_aos, void *slot_image_dst, size_t *slot_bytes_out);

/* moe_unpack_expert — host: slot image -> canonical tensors (the inverse of pack). */
int moe_unpack_expert(int qtype, int H, int F, const void *slot_image, void *gate_aos,
                      void *up_aos, void *down_aos);

/* ------------------------------------------------------------ slot pool (a3) */

/*
 * One expert slot pool for a type/shape group of layers (page 4: groups by tensor
 * type and shape; one VRAM pool per group; LRU shared across the group's layers).
 */
typedef struct {
    int qtype, H, F;
    int n_layers;                     /* layers of this group */
    int n_experts;                    /* routed experts per layer (E) */
    int first_layer;                  /* global index of the group's first layer */
    int n_slots;                      /* slots in the pool */
    size_t slot_bytes;                /* per-slot stride in the pool, >= image bytes, %256 == 0 */
    void *device_pool;                /* device, n_slots * slot_bytes, caller-owned */
    const void *const *host_images;   /* host array [n_layers * n_experts] of pinned slot
                                         images (moe_pack_expert output), layer-major */
    moe_stream_t copy_stream;         /* stream for miss uploads (caller-owned) */
    int device_managed;               /* 0: LRU on the host (moe_cache_ensure); 1: LRU state in
                                         device memory, run on the GPU by moe_cache_plan */
    void *device_state;               /* device_managed: moe_cache_state_bytes() bytes of device
                                         memory, caller-owned, initialised by moe_cache_create */
    size_t device_state_bytes;
    /* Policy variants (0 = off: plain LRU).
     * admit_after: frequency admission (page 3, section "2.2 第二层专家缓存层": experts are
     *   moved into VRAM once their access count passes a threshold).  Every request counts
     *   one access per distinct (layer, expert); a miss whose count, this access included,
     *   is below admit_after takes no slot and changes no LRU state ("bypassed": its slot
     *   is reported as -1 and its weights are read from its pinned host image, see
     *   moe_expert_ffn_fill); it still counts as a miss.  Values 0 and 1 mean plain LRU.
     * lru_window: W tokens (page 1, section 4.3, --moe-lru-window: an expert not used within
     *   the last W tokens is unloaded).  The pool's token clock advances by the ubatch's
     *   token count at every request for the group's first layer; before each request every
     *   slot whose last use is more than W tokens behind the clock is freed.  Host-managed
     *   pools only (MOE_ERR_UNSUPPORTED at create for a device-managed pool). */
    int admit_after;
    int lru_window;
} moe_cache_desc;

typedef struct moe_cache moe_cache; /* opaque, library-owned host object */

typedef struct {
    uint64_t queries[2];      /* distinct (layer, expert) lookups; [0]: ubatch <= 8 tokens, [1]: 9..32 */
    uint64_t hits[2];
    uint64_t misses[2];
    uint64_t evictions;
    uint64_t h2d_bytes;       /* bytes uploaded for misses */
    uint64_t route_queries;   /* per-route (token, expert) lookups */
    uint64_t route_hits;
    uint64_t ensure_calls;
    uint64_t bypassed;        /* misses served from host memory without a slot (admit_after) */
    uint64_t window_evictions;/* slots freed by the LRU window */
    uint64_t prefetch_queries;/* speculative requests (moe_cache_prefetch_plan): distinct experts */
    uint64_t prefetch_hits;   /*   already resident */
    uint64_t prefetch_fills;  /*   given a slot and copied by moe_cache_prefetch_fill */
    uint64_t prefetch_aborts; /*   requests abandoned (more slots than the pool has, or a victim
                                    that the last real request uses) */
} moe_cache_stats;

/*
 * moe_cache_create — validates the descriptor (every host image must be pinned:
 * MOE_ERR_INVALID otherwise; n_slots must be >= 1) and creates an empty pool.
 */
int moe_cache_create(const moe_cache_desc *desc, moe_cache **out);

/*
 * moe_cache_ensure — make the experts of one request resident (host call).
 * ids_host [n_tokens][k] are one layer's routed expert ids.  For the distinct ids,
 * taken in ascending order: hits first (stamped most-recent), then misses, each
 * taking the lowest free slot, else evicting the least-recently-used slot whose
 * expert is not in this request (page 1 section 3.2; page 4).  Each miss is an
 * async cudaMemcpyAsync of the pinned image into its slot on desc.copy_stream,
 * issued after the slot's last reader (see moe_cache_release) has finished.
 * Outputs: slots_host_out [n_tokens*k] (the slot of each input id; -1 for an expert the
 * admission policy bypassed), *n_miss_out (uploads issued), miss_mask_host_out (optional,
 * [n_experts] bytes: 1 for experts uploaded by this call, 0 otherwise), and the layer's
 * device expert->slot table d_slot_table [n_experts] (-1 for non-resident experts),
 * written on stream s.
 * Errors: MOE_ERR_CAPACITY when distinct ids > n_slots (nothing changes);
 * MOE_ERR_INVALID for a layer outside the group or an id outside [0, E);
 * MOE_ERR_CUDA if an upload could not be issued (the slot being filled is left
 * empty and the pool stays consistent).
 */
int moe_cache_ensure(moe_cache *c, int layer, const int32_t *ids_host, int n_tokens, int k,
                     int32_t *slots_host_out, int *n_miss_out, uint8_t *miss_mask_host_out,
                     int32_t *d_slot_table, moe_stream_t s);

/*
 * Device-managed pools (desc.device_managed = 1).  The same pool and the same rules as
 * moe_cache_ensure (page 4's LRU slot pool; page 1 section 3.2's "least-recently-used,
 * not active" victim), with the bookkeeping on the GPU so that a decode step needs no
 * host round trip per layer: the ids never leave the device.
 *
 * moe_cache_state_bytes — device bytes of the state of a pool (slot table, recency list,
 * owners, host image addresses, statistics); the caller allocates it.
 *
 * moe_cache_plan — stream-ordered on s, one CTA: reads the layer's routed ids d_ids
 * [n_tokens][k] (device), applies the LRU rules to the device state and writes
 *   d_table_out [n_experts]  slot of each expert of the layer (-1: not resident),
 *   d_fill_src_out [n_experts] for each expert that missed, the address of its pinned
 *                  host image (the slot it was given must be filled from there), else 0.
 * It moves no weight bytes: moe_expert_ffn_fill reads the missed experts from host memory
 * and writes them into their slots while computing (an expert bypassed by the admission
 * policy gets table -1 and its image address: read from host memory, written nowhere).
 * Capacity overflow or an id out of range is recorded in the device status word
 * (moe_device_status); the layer's table is
 * then all -1 and nothing is read.  Host-side ensure/wait/release are invalid on a
 * device-managed pool; moe_cache_stats_get, moe_cache_lookup and moe_cache_reset work on
 * both kinds (synchronously for this one).
 */
int moe_cache_state_bytes(int n_layers, int n_experts, int n_slots, size_t *bytes);
int moe_cache_plan(moe_cache *c, int layer, const int32_t *d_ids, int n_tokens, int k,
                   int32_t *d_table_out, uint64_t *d_fill_src_out, moe_stream_t s);

/*
 * Cross-layer speculative prefetch for device-managed pools (page 3, tiered MoE scheduling
 * note, section "2.3 第三层传输与计算重叠层": a background stream prefetches the experts
 * the next one or two layers will use while the GPU computes the current layer; section
 * 4.3: prefetch depth 2).
 * moe_cache_prefetch_plan — a speculative request: the same LRU rules as moe_cache_plan for
 *   the predicted ids d_ids [n_tokens][k] of `layer` (hits stamped most recent, misses given
 *   a slot), so the real request later finds them resident; its lookups are counted in the
 *   prefetch statistics, not the hit rate.  It is abandoned (nothing changes, the table is
 *   all -1 and the fill sources 0) if it would need a slot of the last real request of the
 *   pool (that layer's kernels may still be using it) or more slots than the pool has.
 *   Outputs as moe_cache_plan (d_fill_src_out: the image of each expert given a slot).
 * moe_cache_prefetch_fill — copies every expert with d_fill_src[e] != 0 from its pinned host
 *   image into slot d_table[e] (stream-ordered on s; typically a side stream forked after
 *   the plan and joined before the predicted layer's FFN).  The experts' slots must not be
 *   read before the copy completes.
 */
int moe_cache_prefetch_plan(moe_cache *c, int layer, const int32_t *d_ids, int n_tokens, int k,
                            int32_t *d_table_out, uint64_t *d_fill_src_out, moe_stream_t s);
int moe_cache_prefetch_fill(moe_cache *c, const int32_t *d_table, const uint64_t *d_fill_src, moe_stream_t s);

/* moe_cache_wait_uploads — stream s waits for the uploads issued by the last ensure. */
int moe_cache_wait_uploads(moe_cache *c, moe_stream_t s);

/*
 * moe_cache_release — records, on stream s, the point after which the slots of the
 * last ensure are no longer read; later uploads into those slots wait for it.
 * Call it after enqueueing the kernels that read the slots.
 */
int moe_cache_release(moe_cache *c, moe_stream_t s);

int moe_cache_stats_get(const moe_cache *c, moe_cache_stats *out);
/* Clears the pool (all slots empty), the clock and the statistics. Host only. */
int moe_cache_reset(moe_cache *c);
void moe_cache_destroy(moe_cache *c);
/* Slot of (layer, expert) or -1 (host query; for tests). */
int moe_cache_lookup(const moe_cache *c, int layer, int expert);

/*
 * moe_slots_for_budget — slot count per group from a byte budget (page 4, section
 * "配置之前，先算清楚你的专家有多大": budget / per-expert bytes, shared by the groups'
 * layers).  Every group gets n = floor(budget / sum_g per_expert_bytes[g]) slots.
 * A group with fewer than k+1 slots is under budget; if every group is, returns
 * MOE_ERR_BUDGET (page 4: the server refuses to start).
 */
int moe_slots_for_budget(size_t budget_bytes, const size_t *per_expert_bytes, int n_groups,
                         int k, int *slots_out);

/* ------------------------------------------------------ expert FFN (a4..a7, a9) */

/*
 * moe_expert_ffn — the routed experts' SwiGLU FFNs for T tokens, weighted.
 *   for each route (t, j) with e = ids[t][j] (restricted to expert_subset if given):
 *     h = silu(Wg_e x_t) * (Wu_e x_t),   partial[t][j][:] = weights[t][j] * (Wd_e h)
 * Routes of experts outside the subset leave partial[t][j] untouched.
 * x            device [T][H] fp32 or bf16.
 * ids, weights device [T][k] (as produced by moe_router_topk).
 * d_slot_table device [E] int32: expert -> slot in pool (or NULL: slot = expert).
 * pool         device slot images (moe_pack_expert layout), slot s at pool + s*slot_bytes;
 *              pool and slot_bytes must be 16-byte aligned.
 * expert_subset device int32 list of experts to process, or NULL for all.
 * partial      device [T][k][H] fp32 out.
 * workspace    device scratch of moe_expert_ffn_workspace() bytes (256-byte aligned).
 * Path: T <= MOE_DECODE_MAX_T uses the dequantising GEMV kernels (fp32 arithmetic).  Larger
 * T with bf16 activations and H, F multiples of 128 uses the prefill grouped GEMM on tcgen05
 * tensor cores with fp16 operands (activations, dequantised weights d*q[+m] and SwiGLU
 * output each rounded once to fp16) and fp32 accumulation; otherwise the GEMV kernels.
 */
int moe_expert_ffn(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k,
                   const int32_t *ids, const float *weights, const int32_t *d_slot_table,
                   int n_slots, const void *pool, size_t slot_bytes,
                   const int32_t *expert_subset, int n_subset, float *partial,
                   void *workspace, size_t ws_bytes, moe_stream_t s);

/*
 * moe_expert_ffn_fill — moe_expert_ffn over every routed expert, for a device-managed pool:
 * each expert e with d_fill_src[e] != 0 (set by moe_cache_plan for the experts that
 * missed) has its weights read from that pinned host image over the CPU-GPU link and
 * written into its slot (d_slot_table[e]) by the same kernels that compute with them,
 * so the upload and the compute overlap and no copy engine is involved; with
 * d_slot_table[e] == -1 the image is only read (an expert the admission policy bypassed);
 * other experts are read from their slots.  Decode path only (T <= MOE_DECODE_MAX_T or fp32 x);
 * otherwise MOE_ERR_UNSUPPORTED.  The pool must be the one the plan was made for.
 */
int moe_expert_ffn_fill(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k,
                        const int32_t *ids, const float *weights, const int32_t *d_slot_table,
                        int n_slots, void *pool, size_t slot_bytes, const uint64_t *d_fill_src,
                        float *partial, void *workspace, size_t ws_bytes, moe_stream_t s);

/* Workspace bytes of moe_expert_ffn for these sizes (it depends on the path taken). */
int moe_expert_ffn_workspace(int T, int H, int F, int qtype, int xtype, int E, int k, size_t *bytes);

/*
 * moe_expert_ffn_noalloc — moe_expert_ffn for callers that cannot allocate device
 * memory (the pages have no counterpart; this is a library convenience).  Examples: a
 * plugin whose host framework owns every device allocation and passes it only its
 * input and output buffers, or a decode loop where a cudaMalloc/cudaFree, which can
 * synchronise the whole device, is not allowed.  Same arguments and results as
 * moe_expert_ffn, without workspace/ws_bytes; it allocates nothing.
 * Scratch: one array of MOE_NOALLOC_SCRATCH_MAX bytes in device memory, defined in
 * the library, present on every device that loads the library until the process
 * exits.  A request whose moe_expert_ffn_workspace() size exceeds it is rejected with
 * MOE_ERR_UNSUPPORTED before anything is enqueued.
 * Set-up: the first call on a device looks up the array's device address (with that
 * device current) and caches it.  With lazy module loading (the CUDA default) that first
 * call may also load the library's device code and back the array, a one-time cost; so
 * make it during set-up, before any stream capture or latency-critical loop.  A call with
 * T = 0 and valid sizes does only this set-up (x, ids, weights, pool, partial may be NULL).
 * Sharing: every call on a device uses the same array, which keeps the last call's
 * contents (nothing in it needs to start at zero).  Calls whose kernels can overlap on
 * the GPU — different streams, or different host threads — race on the array;
 * serialise them on one stream.
 */
#define MOE_NOALLOC_SCRATCH_MAX (8u << 20)
int moe_expert_ffn_noalloc(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k,
                           const int32_t *ids, const float *weights, const int32_t *d_slot_table,
                           int n_slots, const void *pool, size_t slot_bytes,
                           const int32_t *expert_subset, int n_subset, float *partial,
                           moe_stream_t s);

/* ---------------------------------------------------------------- combine (a8) */

/*
 * moe_combine — y[t][:] = extra[t][:] + sum_{j=0..k-1} partial[t][j][:], summed in the
 * fixed order j = 0..k-1 after extra.  extra (device [T][H] fp32) may be NULL; it
 * carries the residual stream and/or the shared experts' output.  y may alias extra.
 */
int moe_combine(const float *partial, int T, int k, int H, const float *extra, float *y,
                moe_stream_t s);

/*
 * moe_combine_rmsnorm — the combine of a stack layer plus the next layer's input:
 *   y[t]  = extra[t] + sum_{j=0..k-1} partial[t][j]      (as moe_combine; k may be 0)
 *   xn[t] = y[t] / sqrt(mean_h y[t][h]^2 + eps)          (RMS normalisation, unit weight)
 * The pages put the expert FFN inside each transformer block (page 1, section 3.1) but
 * fix no normalisation; the stacks here normalise each layer's input (pre-norm) so that
 * every layer sees inputs of the unit scale the workloads draw.  y or xn may be NULL (not
 * both); xn may not alias y or extra; y may alias extra.  One CTA per token, reductions in
 * a fixed order (deterministic).
 */
int moe_combine_rmsnorm(const float *partial, int T, int k, int H, const float *extra, float *y,
                        float *xn, float eps, moe_stream_t s);

/* ------------------------------------------------------------ device status */

/*
 * moe_device_status — synchronous: reads (and if clear != 0 resets) the current
 * device's status word: MOE_OK, MOE_ERR_INVALID (an id/slot out of range met on
 * the device) or MOE_ERR_TIMEOUT (a bounded wait ran out).  Waits for the device.
 */
int moe_device_status(int *status_out, int clear);

/* ------------------------------------------------------- decode-step runtime */

/*
 * A stack of MoE layers with a pre-norm residual, h_{l+1} = h_l + MoE_l(RMSNorm(h_l))
 * (RMSNorm with unit weight, eps 1e-6; see moe_combine_rmsnorm).  Per layer, by pool kind:
 *  - host-managed pools: router -> ids to the host (one host synchronisation) -> slot-pool
 *    ensure -> FFN over hit experts while misses upload -> FFN over missed experts ->
 *    combine;
 *  - device-managed pools: router -> moe_cache_plan -> moe_expert_ffn_fill -> combine, all
 *    stream-ordered on the GPU with no host round trip;
 *  - every expert resident (n_groups == 0): router -> FFN -> combine, also host-free.
 */
typedef struct {
    int qtype, H, F, E, k, n_layers, n_shared;
    const uint16_t *const *w_router;  /* host array [n_layers] of device [H][E] fp16 */
    const float *const *bias;         /* host array [n_layers] of device [E] fp32, or NULL */
    int n_groups;                     /* slot pools; 0 = every expert resident */
    moe_cache *const *caches;         /* [n_groups]; group g covers its desc's layers */
    const void *resident_pool;        /* n_groups == 0: slot (layer*E + e) images */
    const void *shared_pool;          /* n_shared > 0: slot (layer*n_shared + s) images */
    size_t slot_bytes;                /* slot stride of resident_pool / shared_pool */
    int max_T;                        /* largest ubatch (<= MOE_DECODE_MAX_T) */
    void *workspace;                  /* device, moe_stack_workspace() bytes */
    size_t ws_bytes;
    int overlap;                      /* 1: hit experts run while misses upload */
    int profile;                      /* 0: off; 1: events around the gate/up GEMV only;
                                         2: events around every kernel (moe_stack_profile) */
    int device_managed;               /* 1: the caches are device-managed; each layer runs
                                         router -> moe_cache_plan -> moe_expert_ffn_fill ->
                                         combine on the stream, with no host round trip */
    int use_graph;                    /* device-managed or resident stacks: moe_stack_decode
                                         captures the whole step once per batch size into a
                                         CUDA graph and replays it (inputs/outputs copied in
                                         and out) */
    float load_threshold;             /* 0: off; else routes below it are dropped before the
                                         pools see them (moe_router_topk_threshold; this
                                         changes the layer's output) */
    int prefetch_depth;               /* device-managed pools: 0 off, 1 or 2 = cross-layer
                                         speculative prefetch (page 3, sections 2.3 and 4.3):
                                         after layer l's plan, layers l+1 .. l+depth are routed
                                         on layer l's input, planned speculatively
                                         (moe_cache_prefetch_plan) and their predicted misses
                                         copied into their slots on a side stream while layer l
                                         computes; joined before layer l+1's plan (the plans)
                                         and FFN (the copies).  Values are unchanged. */
} moe_stack_desc;

typedef struct moe_stack moe_stack;

typedef struct {
    uint64_t steps, layers;
    double router_ms, permute_ms, gateup_ms, down_ms, combine_ms; /* summed event times */
    uint64_t gateup_launches, down_launches;
    double gateup_bytes, down_bytes;    /* algorithmic expert bytes streamed */
    double host_wait_ms;                /* host time blocked on the ids readback */
    uint64_t kernel_launches;           /* libmoe kernels launched (counted with or without profile) */
    uint64_t h2d_copies;                /* miss uploads issued */
} moe_stack_profile;

int moe_stack_workspace(int H, int F, int qtype, int E, int k, int max_T, int n_shared,
                        size_t *bytes);
int moe_stack_create(const moe_stack_desc *desc, moe_stack **out);
/*
 * moe_stack_decode — one decode step of T tokens through every layer.
 * x_in, y_out: device [T][H] fp32 (may alias).  With host-managed pools the call
 * synchronises the host once per layer (the slot pools need the routed ids on the host);
 * with device-managed pools or a resident stack it only enqueues work on s (and with
 * use_graph replays a captured step).  All kernels run on s.
 * ids_host_out / weights_host_out (optional, host [n_layers][T][k]) receive the routing
 * (valid once s has completed; such a call is never graph-replayed).
 */
int moe_stack_decode(moe_stack *st, const float *x_in, float *y_out, int T,
                     int32_t *ids_host_out, float *weights_host_out, moe_stream_t s);
/* moe_stack_layer — one layer only: y = x + MoE_layer(x) (same semantics as decode). */
int moe_stack_layer(moe_stack *st, int layer, const float *x_in, float *y_out, int T,
                    int32_t *ids_host_out, float *weights_host_out, moe_stream_t s);
/* Synchronises the stream of the last call and returns the accumulated profile. */
int moe_stack_profile_get(moe_stack *st, moe_stack_profile *out);
int moe_stack_profile_reset(moe_stack *st);
/* Sets the profiling level (0, 1, 2 as in moe_stack_desc.profile) for later calls. */
int moe_stack_set_profile(moe_stack *st, int level);

/*
 * moe_stack_gemv_timing — the decode GEMV kernels of a resident stack (n_groups == 0)
 * timed alone: the router and the token-to-expert permute of every layer run first for the
 * batch x_in (device [T][H] fp32, the same FFN input for each layer, 1 <= T <=
 * MOE_DECODE_MAX_T); then, on stream s behind a GPU spacer (a bounded spin, so that every
 * timed launch is queued before the first starts), `reps` rounds of the gate/up GEMV of
 * every layer are launched back to back between two CUDA events, then `reps` rounds of the
 * K-split reduce (if any), then `reps` rounds of the down GEMV, then `reps` rounds of the
 * whole decode FFN chain of every layer as the FFN entry points run it: the permute kernel,
 * then the fused GEMV launch when moe_get_decode_fused() is 1, else the three GEMV kernels.
 * Consecutive launches read different layers' experts, so no launch finds the previous
 * one's weights in L2.  Results: the average time of one launch (microseconds, launch gaps
 * included, no events between launches) and the quantised bytes of the selected experts
 * one launch reads (the permute kernel's active-expert counts).  Allocates and frees its
 * own device buffers and synchronises s.  Errors: MOE_ERR_UNSUPPORTED for a stack with
 * pool groups.
 */
typedef struct moe_gemv_timing {
    double gateup_us, down_us;        /* average per launch */
    double gateup_bytes, down_bytes;  /* average per launch */
    int launches;                     /* per kernel: reps * layers */
    double reduce_us;                 /* the K-split reduce between them (0 launches when the
                                         gate/up GEMV does not split K), timed the same way */
    double gemv_us;                   /* one layer's whole chain: permute, gate/up, reduce, down */
    int fused;                        /* 1: gemv_us timed the fused GEMV launch */
} moe_gemv_timing;
int moe_stack_gemv_timing(moe_stack *st, const float *x_in, int T, int reps, moe_gemv_timing *out,
                          moe_stream_t s);
void moe_stack_destroy(moe_stack *st);

/*
 * moe_set_decode_fused — process-wide choice of how the decode path runs its GEMVs.
 * on == 0 (the default): the gate/up GEMV, the K-split reduce and the down GEMV run as
 * three kernels one after another.  on != 0: as one cooperative launch whose CTAs meet at a
 * grid barrier (bounded wait: MOE_ERR_TIMEOUT in the status word) after issuing their
 * down-weight copies, so that the down GEMV's weight reads overlap the gate/up GEMV's tail
 * (measured slower on GB300 at the decode sizes: each grid barrier costs about as much as a
 * launch).  Both compute the same values in the same order.  Takes effect for calls (and
 * graph captures) made after it; a captured graph keeps the choice it was captured with.
 */
int moe_set_decode_fused(int on);
int moe_get_decode_fused(void);

/* ------------------------------------------------------------------ test hooks */

/*
 * moe_debug_inject_fault — fault injection for tests, armed on the host; kind 0 disarms.
 *  kind 1: the n-th following miss upload (n = countdown, 0 = the next) fails as if the
 *          copy could not be issued.  Never touches the GPU.
 *  kind 2: the n-th following fused decode GEMV launch (moe_set_decode_fused(1)) is given
 *          a grid barrier that waits for one arrival more than it has CTAs, bounded at
 *          20 ms: every CTA's wait runs out, MOE_ERR_TIMEOUT is recorded in the device status
 *          word and the kernel goes on to its end (its outputs are then meaningless).  This
 *          exercises the bounded-wait path without faulting or hanging the GPU.
 */
int moe_debug_inject_fault(int kind, int countdown);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
