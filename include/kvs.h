/*
 * kvs.h -- host-streamed, block-paged, quantised KV attention on one GB300.
 *
 * The complete KV history of every layer lives in host memory (pinned, or
 * registered by kvs_create).  A bounded device arena holds resident pages of
 * chosen layers plus a single transfer ring that every layer uses; a copy stream
 * refills ring slots from host memory ahead of the attention stream, fenced
 * by a "ready" event (attention waits for the copy) and a "consumed" event
 * (the next copy into a slot waits for its last reader), and every layer
 * still attends over its complete history.  Design source: "Adaptive KV
 * Streaming for llama.cpp V2" (sections "KV data movement and attention",
 * "Keep the stock attention order", "Backend-neutral memory and streaming
 * contracts") and "Adaptive KV Streaming for llama.cpp" (section "Adaptive KV
 * streaming": resident pages plus one shared ring, consumed slots recycled
 * immediately, the full history still attended).
 *
 * Cache types: K uses Q8_0 and V uses Q4_0 (32-element blocks, fp16 scale), the
 * one K/V pairing the pages qualify for streaming.  Other
 * types are refused (KVS_ERR_UNSUPPORTED), as the pages require a backend to
 * advertise only the K/V pairs it really supports.
 *
 * Conventions shared by every entry point:
 *  - Every call returns a kvs_status; nothing aborts, throws or traps.  On
 *    failure kvs_last_error(ctx) holds a one-line reason (valid until the
 *    next call on that context).  Errors are returned rather than aborting
 *    because a too-tight arena or an oversize batch must be an error return
 *    (PR "port adaptive KV streaming", review comments).
 *  - The library allocates no device or host memory: the caller owns the
 *    arena, the workspace, the host history, Q, out and lse, and keeps them
 *    alive until kvs_destroy.  It creates CUDA events and two streams of its
 *    own: one for reads of resident pages (lowest priority) and one for lane
 *    0's ring reads.
 *  - All device work is ordered with respect to the caller's streams
 *    (attn_stream, copy_stream and the lanes' streams): the library's own
 *    streams fork from them by events and join back into attn_stream before
 *    the combine.  Calls return once work is enqueued; results are valid
 *    after the attention stream reaches that point (kvs_sync, or any later
 *    work on attn_stream).
 *  - A context serves one sequence and is not thread-safe.
 *  - Sizes and layouts use these symbols: P = page_tokens, Hk = n_kv_head,
 *    D = head_dim, Hq = query heads (a multiple of Hk; query head h reads kv
 *    head h / (Hq / Hk)), T = tokens appended to a layer.
 */
#ifndef KVS_H_
#define KVS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVS_ABI_VERSION 4

typedef struct kvs_ctx kvs_ctx;

typedef enum {
    KVS_OK = 0,
    KVS_ERR_INVALID = -1,     /* bad argument or call order */
    KVS_ERR_UNSUPPORTED = -2, /* geometry or type the library does not serve */
    KVS_ERR_ARENA = -3,       /* arena or workspace below the minimum */
    KVS_ERR_HOST = -4,        /* host history too small or cannot be registered */
    KVS_ERR_CUDA = -5,        /* a CUDA runtime call failed (message in last_error) */
    KVS_ERR_COVERAGE = -6,    /* the span plan would leave a gap or overlap */
    KVS_ERR_CAPACITY = -7,    /* beyond max_tokens, the resident pool, or appended length */
    KVS_ERR_TIMEOUT = -8,     /* kvs_sync deadline passed */
    KVS_ERR_INJECTED = -9,    /* a fault armed by kvs_debug_inject fired */
    KVS_ERR_STATE = -10       /* call not allowed in the current state (e.g. pending prefetch) */
} kvs_status;

/* Block types, numbered as the ggml type ids of the same formats. */
typedef enum { KVS_TYPE_Q4_0 = 2, KVS_TYPE_Q8_0 = 8 } kvs_qtype;
/* Query element types accepted by kvs_attend. */
typedef enum { KVS_F32 = 0, KVS_F16 = 1 } kvs_dtype;

/* kvs_config.flags */
#define KVS_FLAG_PLAN_ONLY 1u /* host scheduling only: no CUDA call is made, no
                                 kernel runs and no output is written; every
                                 operation the context would enqueue is logged
                                 for kvs_trace_read.  For testing the host-side
                                 planner on machines without a GPU. */
#define KVS_FLAG_DMA_FILL 2u  /* ring refills and pool loads by the copy engines
                                 (one cudaMemcpyAsync per run of pages that are
                                 consecutive in both host and device memory)
                                 instead of the SM-driven fill kernel: no SM
                                 time, a fixed cost per copy */
#define KVS_FLAG_F16_OPERANDS 4u /* split-K attention (decode, span verify) feeds the
                                 tensor cores the query and the softmax weights
                                 times the V scale as single f16 values (about 11
                                 significant bits) instead of f16 hi + lo pairs
                                 (about 22): half the MMAs, measured relative
                                 error ~5e-4 instead of ~1e-6 against the fp64
                                 oracle; accumulation stays fp32 */

typedef struct {
    uint32_t page_tokens;  /* P: token positions per page; 32, 64, 128 or 256 */
    uint32_t n_layers;     /* attention layers, each with its own history */
    uint32_t n_kv_head;    /* Hk */
    uint32_t head_dim;     /* D: 64, 128 or 256 */
    uint32_t max_q_head;   /* upper bound on Hq (multiple of Hk); sizes the workspace */
    uint32_t max_rows;     /* upper bound on query rows per kvs_attend; sizes the workspace */
    uint64_t max_tokens;   /* history capacity per layer, tokens */
    int32_t k_type;        /* KVS_TYPE_Q8_0 */
    int32_t v_type;        /* KVS_TYPE_Q4_0 */
    void *arena;           /* device bytes for page slots: 2 tail slots per layer,
                              the resident pool and the ring; 256-byte aligned */
    uint64_t arena_bytes;
    void *workspace;       /* device bytes for split-K partials; 256-byte aligned */
    uint64_t workspace_bytes;
    void *host;            /* host history: n_layers * ceil(max_tokens/P) pages, layer-major;
                              registered with CUDA by kvs_create if not already pinned.
                              Prefer memory from cudaHostAlloc: ring refills read it
                              through the GPU's mappings, and registered pageable memory
                              is mapped with small pages (on GB300 a 27 GB registered
                              history streamed at 7.5 % of the link, a cudaHostAlloc one
                              at 89 %) */
    uint64_t host_bytes;
    uint32_t ring_slots;   /* initial ring size in page slots (>= 1) */
    uint32_t chunk_pages;  /* ring pages per ready/consumed handshake; 0: ring_slots/4
                              clamped to 1..32 */
    void *attn_stream;     /* cudaStream_t for attention, quantise/append and pool moves */
    void *copy_stream;     /* cudaStream_t for ring refills, pool loads and D2H publish */
    uint32_t flags;        /* KVS_FLAG_* */
    uint32_t n_lanes;      /* ring pipelines, 1..8 (0 = 1): ring chunk j is copied on copy
                              lane j % n_lanes and attended on attention lane j % n_lanes, so
                              neighbouring chunks' copies and reads overlap; lane 0 is
                              (attn_stream, copy_stream) */
    void *lane_attn_streams[7];  /* cudaStream_t of attention lanes 1 .. n_lanes-1 */
    void *lane_copy_streams[7];  /* cudaStream_t of copy lanes 1 .. n_lanes-1 */
    uint32_t prefill_split_pages; /* pages per split of the tensor-core prefill path (0 = 24,
                                     at most ring_slots and at most 128); when max_q_head *
                                     max_rows allows that path, ring chunks never cross a
                                     split.  Longer splits write fewer partials and spend
                                     less of each CTA on its prologue and epilogue */
    uint32_t max_verify_rows;     /* widest kvs_attend (query rows) served on the split-K
                                     kernel; calls beyond 64 rows x heads per kv head run as
                                     row groups and need workspace for every row: 0 = max_rows
                                     when the geometry has no tensor-core prefill path, else
                                     64 / (max_q_head / n_kv_head) rows (no row groups) */
} kvs_config;

typedef struct {
    uint64_t h2d_bytes;        /* ring refill bytes copied host -> device */
    uint64_t h2d_pages;        /* ring refill pages */
    uint64_t h2d_launches;     /* ring refill copy launches (one per chunk) */
    uint64_t pool_load_bytes;  /* host -> resident pool bytes (kvs_set_residency) */
    uint64_t d2h_bytes;        /* tail pages published device -> host */
    uint64_t d2h_pages;
    uint64_t ring_chunks;      /* ring chunks attended (ready/consumed handshakes) */
    uint64_t ring_recycles;    /* ring slot refills that reused a previously read slot */
    uint64_t resident_pages_read;  /* page-head items read from pool or tail slots */
    uint64_t ring_pages_read;      /* page-head items read from ring slots */
    uint64_t attend_calls;
    uint64_t kernel_launches;  /* kernels this context launched (all kinds) */
    uint64_t decode_launches;  /* split-K attention kernel launches */
    double decode_ms;          /* summed device time of timed attention launches (kvs_set_timing) */
    uint64_t decode_timed;     /* number of attention launches in decode_ms */
    uint64_t decode_bytes;     /* page bytes those timed launches read (items * page_bytes) */
    uint64_t ring_slots;       /* current ring size */
    uint64_t pool_slots;       /* current resident pool size */
    uint64_t pool_used;        /* pool slots holding a resident page */
    uint64_t graph_launches;   /* kvs_graph_launch calls */
    uint64_t graph_kernels;    /* kernels in the captured step graph */
    uint64_t chunk_pages;      /* current ring chunk size, pages */
    /* the policy's feedback as the last kvs_observe measured it (see there) */
    uint64_t observed_reads;   /* ring chunk reads accounted */
    uint64_t ready_misses;     /* of those, reads that waited for their copy */
    double ring_occupancy;     /* mean fraction of ring slots holding a page not yet read */
    double copy_busy;          /* fraction of the interval the refills were running */
} kvs_stats_t;

/* One logged operation of a KVS_FLAG_PLAN_ONLY context (see kvs_trace_read). */
typedef struct {
    uint32_t op;      /* KVS_OP_* */
    uint32_t stream;  /* 2*lane: attention stream of that lane, 2*lane+1: its copy stream */
    uint32_t layer;
    uint32_t event;   /* event id (RECORD / WAIT) */
    int64_t a;        /* READ/FILL/POOL_LOAD/PUBLISH/WRITE: page; LAUNCH: kernel kind */
    int64_t b;        /* READ/FILL/POOL_LOAD/PUBLISH/WRITE: device slot; LAUNCH: items */
    int64_t c;        /* READ: kv head; FILL: ring sequence number */
    int64_t d;        /* reserved */
} kvs_trace_op;

enum {
    KVS_OP_RECORD = 1,    /* record event `event` on `stream` */
    KVS_OP_WAIT = 2,      /* `stream` waits for the last record of `event` */
    KVS_OP_FILL = 3,      /* copy stream: host page a -> ring slot b */
    KVS_OP_READ = 4,      /* attention kernel reads page a (kv head c) from slot b */
    KVS_OP_POOL_LOAD = 5, /* copy stream: host page a -> pool slot b */
    KVS_OP_PUBLISH = 6,   /* copy stream: slot b -> host page a (D2H) */
    KVS_OP_WRITE = 7,     /* attention stream: new rows quantised into page a in slot b */
    KVS_OP_LAUNCH = 8,    /* a kernel launch of kind a over b items */
    KVS_OP_MOVE = 9       /* attention stream: device copy of page a into pool slot b */
};

/* kvs_debug_inject fault kinds.  None of them makes a GPU fault: each is made
 * on the host, or (KVS_FAULT_DEVICE_WAIT) as a device-side wait that gives
 * up by its own limit and reports a status. */
enum {
    KVS_FAULT_NONE = 0,
    KVS_FAULT_FILL_ENQUEUE = 1, /* the nth ring refill enqueue fails */
    KVS_FAULT_SYNC_STALL = 2,   /* kvs_sync sees the GPU as busy until its deadline */
    KVS_FAULT_DEVICE_WAIT = 3   /* in the split-K attention launches of the nth kvs_attend call,
                                   every pipeline wait gives up at once, as if its copy never
                                   landed: the CTAs drain the copies they issued (with the
                                   normal bound), set the status word and exit.  That call's
                                   outputs (and those of later calls until the next kvs_sync)
                                   are NaN, and the next kvs_sync returns KVS_ERR_CUDA */
};

/*
 * kvs_query_sizes -- sizes a configuration needs.  Fields read: page_tokens,
 * n_layers, n_kv_head, head_dim, max_q_head, max_rows, max_tokens, ring_slots.
 *   page_bytes:      bytes of one page (all kv heads): Hk * P * D * 13 / 8
 *   host_bytes:      minimum host history bytes
 *   arena_bytes_min: minimum arena (2 tail slots per layer + ring_slots)
 *   workspace_bytes: minimum workspace (a 256-byte status word, then split
 *                    partials for max_rows rows)
 * Any output pointer may be NULL.  The page size follows the cache types:
 * per token and kv head, Q8_0 K takes D + 2*D/32 bytes and Q4_0 V takes
 * D/2 + 2*D/32 bytes (V2 README, "KV data movement and attention": page sizes
 * follow the selected quants).
 *
 * Page layout.  A page is Hk head sections of S = P*D*13/8 bytes, kv head g at
 * byte g*S.  With NB = D/32 blocks of 32 dims, token t (0 <= t < P) and dim d,
 * a head section holds four sub-arrays:
 *   Kq  offset 0,           P*D bytes:    the int8 Q8_0 code of (t, d) at byte
 *                            ((t/16*NB + d/32)*16 + t%16)*32 + d%32
 *                            (16-token groups; within a group block-major, then
 *                            token, then the block's 32 codes)
 *   Ks  offset P*D,         P*D/16 bytes: the fp16 Q8_0 scale of (t, block b)
 *                            at fp16 element t*NB + b
 *   Vq  offset P*D*17/16,   P*D/2 bytes:  byte row j (0 <= j < D/2) packs dims
 *                            j/16*32 + j%16 (low nibble) and j/16*32 + j%16 + 16
 *                            (high nibble); the byte of (t, j) is at
 *                            ((t/32*NB + j/16)*16 + j%16)*32 + t%32
 *                            (32-token chunks; within a chunk byte row, then
 *                            the chunk's 32 tokens)
 *   Vs  offset P*D*25/16,   P*D/16 bytes: the fp16 Q4_0 scale of (t, block b)
 *                            at fp16 element b*P + t
 * Values: K = code * scale; V = (nibble - 8) * scale (Q4_0 codes 0..15).
 * fp16 scales are little-endian IEEE binary16.  These orders hand each
 * tensor-core fragment of the attention kernel to one 8-byte load; the codes
 * and scales themselves are exactly the Q8_0 / Q4_0 block contents.
 */
kvs_status kvs_query_sizes(const kvs_config *cfg, uint64_t *page_bytes, uint64_t *host_bytes,
                           uint64_t *arena_bytes_min, uint64_t *workspace_bytes);

/*
 * kvs_create -- validate cfg and build a context.  The arena is carved into
 * page slots: 2 * n_layers tail slots, then ring_slots ring slots, the rest
 * is the resident pool (the device KV budget is the resident pages of all
 * layers plus the ring slots they share: V2 README, "KV data movement and
 * attention").
 * Refusals: geometry outside the supported set or k/v types other than
 * Q8_0/Q4_0 -> KVS_ERR_UNSUPPORTED; arena or workspace below the minimum ->
 * KVS_ERR_ARENA (the pages refuse a too-small arena at start-up); host
 * history too small or not registrable -> KVS_ERR_HOST.  *out is NULL on
 * failure.
 */
kvs_status kvs_create(const kvs_config *cfg, kvs_ctx **out);

/* kvs_destroy -- synchronise the context's streams, release events and any
 * host registration made by kvs_create.  Never frees caller memory (the
 * caller owns the arena: V2 README, "Phase arena": one device-local parent
 * allocation, lent out as bounded views).  Library API otherwise; the pages
 * describe no such call. */
kvs_status kvs_destroy(kvs_ctx *ctx);

/*
 * kvs_append -- the KV writer: quantise n_tokens new rows of layer `layer`
 * (k_dev, v_dev: device fp32 [n_tokens][Hk][D]) into the layer's device tail
 * page(s) at positions T .. T+n_tokens-1 (K -> Q8_0, V -> Q4_0, on
 * attn_stream).  A page that becomes full is published device -> host on the
 * copy stream as soon as it is written (the V2 README publishes a changed
 * tail to host when it is produced); it stays
 * readable on the device until the page after next starts, and then moves to
 * the resident pool if the layer's residency mask asks for it and the pool
 * has room, else it is streamed from host like any other nonresident page.
 * KVS_ERR_CAPACITY if T + n_tokens > max_tokens.
 */
kvs_status kvs_append(kvs_ctx *ctx, uint32_t layer, const float *k_dev, const float *v_dev,
                      uint32_t n_tokens);

/* kvs_truncate -- shorten layer `layer` to n_tokens (<= T), e.g. to drop a
 * rejected draft suffix (V2 README, "MTP catch-up, prediction, and rollback":
 * on rejection the rejected KV suffix is discarded and accepted work kept).
 * Only the current tail page (and the page before it) may be cut into;
 * KVS_ERR_UNSUPPORTED for a cut further back.  KVS_ERR_STATE while the layer
 * has prefetched ring pages pending.  Rows appended afterwards overwrite the
 * tail and publish it to host again once the page is full. */
kvs_status kvs_truncate(kvs_ctx *ctx, uint32_t layer, uint64_t n_tokens);

/* kvs_length -- tokens appended to layer `layer`.  Library API; the pages
 * describe no such call. */
kvs_status kvs_length(const kvs_ctx *ctx, uint32_t layer, uint64_t *n_tokens);

/*
 * kvs_load_host_pages -- write n_pages complete, already encoded pages (src:
 * host memory, n_pages * page_bytes, each in the page layout kvs_query_sizes
 * gives) into the host history of `layer` as pages first_page ..
 * first_page + n_pages - 1, and extend the layer to (first_page + n_pages) * P
 * tokens.  The host history is the authoritative copy of every page (V2
 * README, "KV data movement and attention"), so a history encoded elsewhere
 * can be installed there without passing each row through the KV writer.
 * first_page must equal T / P with T a multiple of P (KVS_ERR_INVALID
 * otherwise), and the pages must fit max_tokens (KVS_ERR_CAPACITY).  The call
 * first waits for the context's earlier device work (a publish may still be
 * writing the host history), then copies on the host; it returns when the
 * bytes are in place.  The loaded pages are host-only: they are streamed
 * through the ring when attended, until a later kvs_set_residency makes some
 * resident.  The tail slots keep the pages they held, so the next kvs_append
 * starts a new page.  KVS_ERR_STATE while prefetches are pending or inside a
 * step capture.
 */
kvs_status kvs_load_host_pages(kvs_ctx *ctx, uint32_t layer, uint64_t first_page, uint64_t n_pages,
                               const void *src);

/*
 * kvs_set_residency -- choose which pages of `layer` live in the resident
 * pool: mask[i] != 0 for page i (i < n_pages; pages >= n_pages are not
 * resident).  Newly resident pages are loaded host -> pool on the copy
 * stream; attention waits for the load before its next read (selected pages
 * go host -> resident pool, and one layer may stay fully resident while
 * others stream: V2 README, "KV data movement and attention").  The device
 * tail pages are always device-readable whatever the mask says.
 * KVS_ERR_CAPACITY if the pool has too few free slots (nothing changes);
 * KVS_ERR_STATE while any layer has prefetched ring pages pending.
 */
kvs_status kvs_set_residency(kvs_ctx *ctx, uint32_t layer, const uint8_t *mask,
                             uint64_t n_pages);

/*
 * kvs_set_ring_slots -- re-split the arena between the resident pool and the
 * ring: ring = n_slots page slots (>= 1), chunk = chunk_pages (0: default).
 * Under pressure the pages' policy trades resident pages for ring slots
 * within one physical budget (V2 README, "KV data movement and attention");
 * the runtime repartitions the pool only once a proposal is accepted ("Logical
 * KV layout, policy, and physical execution").
 * KVS_ERR_CAPACITY if the pool would become smaller than the pages resident
 * now; KVS_ERR_STATE while prefetches are pending.  Waits for earlier ring
 * work on the device (stream-ordered) before slots change role.
 */
kvs_status kvs_set_ring_slots(kvs_ctx *ctx, uint32_t n_slots, uint32_t chunk_pages);

/*
 * Adaptive residency policy (Adaptive KV Streaming for llama.cpp V2, "KV data
 * movement and attention" and "Logical KV layout, policy, and physical
 * execution"; Adaptive KV Streaming for llama.cpp, "Adaptive KV streaming").
 * The pages' policy proposes the resident/ring split of a fixed slot budget
 * from the active context length and from feedback (how many reads waited
 * on a copy, how full the ring ran, how busy the copy stream was), and
 * changes it only after consistent evidence (hysteresis).  It moves no bytes and
 * launches nothing; the caller applies a decision with kvs_set_ring_slots
 * and kvs_set_residency.  The pages give no thresholds; these are the
 * caller's, in kvs_policy_config.
 */
typedef struct {
    uint32_t page_tokens;     /* tokens per page */
    uint32_t n_layers;        /* attended layers sharing the budget */
    uint32_t budget_slots;    /* page slots shared by resident pages and the ring */
    uint32_t min_ring_slots;  /* ring lower bound (>= 1) */
    uint32_t max_ring_slots;  /* ring upper bound (0: budget_slots) */
    uint32_t step_slots;      /* slots moved between pool and ring per change (>= 1) */
    uint32_t hold_steps;      /* consecutive agreeing observations before a change (>= 1) */
    float miss_grow;          /* grow when ready_misses / streamed_reads exceeds this ... */
    float copy_busy_max;      /* ... and the copy stream was busy less than this fraction */
    float occupancy_shrink;   /* shrink when no read missed and the ring held prefetched
                                 pages for less than this fraction of its slots */
    float link_gbs;           /* > 0: the host link's measured copy rate (GB/s); the link
                                 then has room while the observed refill rate
                                 (copy_bytes / interval_ns) is below copy_busy_max times
                                 it, instead of while copy_busy is below copy_busy_max */
} kvs_policy_config;

typedef struct {              /* zero-initialise before the first step */
    uint32_t ring_slots;      /* the split in force (0: none yet) */
    uint32_t grow_run;        /* consecutive observations asking for a larger ring */
    uint32_t shrink_run;      /* consecutive observations asking for a smaller ring */
    uint32_t steps;           /* observations taken */
} kvs_policy_state;

typedef struct {              /* one observation interval, e.g. one decode step */
    uint64_t context_tokens;  /* active history length per layer */
    uint64_t streamed_reads;  /* ring chunk reads in the interval */
    uint64_t ready_misses;    /* of those, reads whose copy had not finished when issued */
    float ring_occupancy;     /* mean fraction of ring slots holding a page not yet read */
    float copy_busy;          /* fraction of the interval the copy stream was busy */
    uint64_t copy_bytes;      /* bytes the interval's refills moved (0: not measured) */
    uint64_t interval_ns;     /* length of the interval (0: not measured) */
} kvs_policy_observation;

enum {
    KVS_POLICY_INIT = 1,      /* first decision: smallest ring */
    KVS_POLICY_FITS = 2,      /* the whole history fits resident: smallest ring */
    KVS_POLICY_HOLD = 3,      /* no change */
    KVS_POLICY_GROW = 4,      /* reads waited on copies while the link had room */
    KVS_POLICY_SHRINK = 5,    /* the ring sat mostly empty and no read waited */
    KVS_POLICY_CLAMP = 6      /* the split in force was outside the bounds */
};

typedef struct {
    uint32_t ring_slots;               /* proposed ring size */
    uint32_t resident_slots;           /* budget_slots - ring_slots */
    uint64_t resident_pages_per_layer; /* min(pages per layer, resident_slots / n_layers) */
    uint64_t pages_per_layer;          /* ceil(context_tokens / page_tokens) */
    uint32_t reason;                   /* KVS_POLICY_* */
    int32_t changed;                   /* ring_slots differs from the previous split */
} kvs_policy_decision;

/*
 * kvs_policy_step -- one policy decision.  Pure host function (no context,
 * no CUDA): reads config, previous state and observation; writes the next
 * state and the decision.  Rules, in order:
 *  1. The whole history (pages per layer x n_layers) fits in budget_slots
 *     minus the smallest ring: smallest ring (FITS); resident space is kept
 *     as large as the budget allows.
 *  2. No split yet: smallest ring (INIT).
 *  3. Otherwise an observation asks to grow when the miss rate exceeds
 *     miss_grow while the link has room (a deeper prefetch helps only then):
 *     with link_gbs > 0 and a measured interval, while copy_bytes /
 *     interval_ns < copy_busy_max x link_gbs, else while copy_busy <
 *     copy_busy_max; and to shrink when no read missed and
 *     ring_occupancy < occupancy_shrink.  A change of step_slots is made
 *     after hold_steps consecutive observations agree; any other observation
 *     restarts the count (hysteresis), and a change restarts both counts.
 *  4. The result is clamped to [min_ring_slots, max ring], where max ring =
 *     min(max_ring_slots or budget_slots, budget_slots).
 * KVS_ERR_INVALID (nothing written) for null pointers, page_tokens,
 * n_layers, budget_slots, step_slots or hold_steps of 0, min_ring_slots of 0
 * or above the max ring, or fractions outside [0, 1].
 */
kvs_status kvs_policy_step(const kvs_policy_config *config, const kvs_policy_state *previous,
                           const kvs_policy_observation *observation, kvs_policy_state *next,
                           kvs_policy_decision *decision);

/*
 * Complete-layer lease and ring guard (V2 README, "MTP catch-up, prediction,
 * and rollback": an attached layer with its own host history borrows the
 * resident/ring pool, loads its nonresident suffix into the ring once for a
 * catch-up and draft phase, and gives the whole ring back afterwards; and
 * "Backend-neutral memory and streaming contracts": the lease holder keeps the
 * ring protected from the other layers' lookahead, and committed tail rows
 * extend the retained lease).
 *
 * kvs_lease_acquire -- take 1 slot per nonresident page of `layer` (pages in
 * neither the pool nor a tail slot), plus extra_slots spare slots, off the top
 * of the ring, and load those pages into them on the copy stream (attention
 * waits for the load).  While the lease is held: attends of `layer` read every
 * page from the device (no ring chunks); the other layers stream through the
 * remaining ring slots, so no refill ever writes a leased slot; a page leaving
 * `layer`'s tail slots moves into a spare slot (while spares remain, else it
 * is treated as usual); a truncation that drops leased pages returns their
 * slots to the spares.  kvs_page_location reports leased pages as kind 3.
 * kvs_set_residency, kvs_set_ring_slots and kvs_load_host_pages are refused
 * (KVS_ERR_STATE) while a lease is held.  Refusals: a lease already held or
 * prefetches pending -> KVS_ERR_STATE; the ring would keep no slot ->
 * KVS_ERR_CAPACITY.  Acquire and release wait for earlier ring work on the
 * device (stream-ordered) and drop a captured step graph.
 *
 * kvs_lease_release -- give every leased slot back to the ring; the pages are
 * host-only again (the host history holds them unchanged).  kvs_lease_info
 * reports the leased layer (-1 if none), the slots it holds and its spares.
 */
kvs_status kvs_lease_acquire(kvs_ctx *ctx, uint32_t layer, uint32_t extra_slots);
kvs_status kvs_lease_release(kvs_ctx *ctx);
kvs_status kvs_lease_info(const kvs_ctx *ctx, int64_t *layer, uint32_t *leased_slots, uint32_t *spare_slots);

/*
 * kvs_observe -- the feedback the residency policy samples (V2 README, "KV
 * data movement and attention": readiness misses, ring occupancy and
 * copy-stream time), measured on the device since the last reset, as a
 * kvs_policy_observation: every ring refill by the SM fill kernel stamps its
 * start and end (%globaltimer), and the read of that chunk accounts, at its
 * start, whether it waited for the copy (it started within 4 us of the copy's
 * end: a readiness miss) and how long the chunk's pages sat in the ring
 * unread.  context_tokens = the longest layer; streamed_reads, ready_misses =
 * chunk reads accounted and missed; ring_occupancy = sum over reads of
 * pages x (read start - copy end) / (interval x ring_slots); copy_busy = sum
 * of copy durations / interval (at most 1; refills of several lanes that
 * overlap each count), the interval running from the first copy's start to
 * the last read's start; copy_bytes = page bytes of the accounted refills;
 * interval_ns = that interval.  Refills by the copy engines
 * (KVS_FLAG_DMA_FILL) are not stamped and not accounted.  Waits for the
 * context's device work first (kvs_sync); reset != 0 starts a new interval.
 * The counters also accumulate across step-graph replays.  The values are
 * copied into kvs_stats_t.  Library API (the pages give the inputs, not a call).
 */
kvs_status kvs_observe(kvs_ctx *ctx, kvs_policy_observation *out, int reset);

/*
 * kvs_prefetch -- announce that `layer` is attended next (after any layer
 * already announced) and enqueue host -> ring copies of its nonresident pages
 * into ring slots whose previous reader has already been enqueued: copies
 * for later layers proceed while the current layer is attended (V2 README,
 * "KV data movement and attention").  Non-blocking; copies that do not
 * fit yet are issued by later kvs_attend calls as slots free up.  Layers must
 * then be attended in announcement order (KVS_ERR_STATE otherwise).
 */
kvs_status kvs_prefetch(kvs_ctx *ctx, uint32_t layer);

/*
 * kvs_attend -- causal attention of n_rows query rows of layer `layer` over
 * its complete history.  q_dev: device [n_rows][n_q_head][D], fp32 or fp16
 * (q_dtype); row r sits at position pos0 + r and sees keys 0 .. pos0 + r
 * (requires pos0 + n_rows <= T: append the rows' own K/V first).  out_dev:
 * device fp32 [n_rows][n_q_head][D], normalised; lse_dev (nullable): device
 * fp32 [n_rows][n_q_head], natural-log sum of exp of the scaled scores.
 * Scores are scale * q . k.
 * Pages are read from their tail/pool slot, or from ring slots filled from
 * host on the copy stream; each ring chunk is attended after its ready event
 * and its slots are released by a consumed event.  The split-K partition is
 * one partial per (page, kv head) whatever the residency, and the final
 * log-sum-exp combine runs over pages in logical order, so the result is
 * bitwise identical for any residency or ring size ("Keep the stock
 * attention order", V2 README).
 * Rows: 1 (decode) up to floor(64 / (Hq/Hk)) (span verify, e.g. 2..6 draft
 * rows with 6 query heads per kv head) run on the split-K kernel with one
 * partial per page.  Wider calls with fp16 queries at head_dim 256 and
 * page_tokens a multiple of 64 (a prefill chunk, up to 256 rows) run on the
 * tcgen05 tensor-core kernel with one partial per prefill split (a fixed
 * group of prefill_split_pages pages, so the result is again independent of
 * residency and ring size).  Any other wider call (e.g. an fp32 ngram verify
 * of 49 rows) runs on the split-K kernel as consecutive row groups of at most
 * 64 rows x heads per kv head, every group reading each staged ring span
 * before its slots are released, with one partial per (page, row, head):
 * n_rows must be <= max_verify_rows (KVS_ERR_UNSUPPORTED otherwise).  A
 * timed-out device-side wait is reported by the next kvs_sync as
 * KVS_ERR_CUDA.
 */
kvs_status kvs_attend(kvs_ctx *ctx, uint32_t layer, const void *q_dev, int32_t q_dtype,
                      uint32_t n_rows, uint32_t n_q_head, uint64_t pos0, float scale,
                      float *out_dev, float *lse_dev);

/* kvs_sync -- wait until every stream of the context has finished its work,
 * or return KVS_ERR_TIMEOUT after timeout_ms (0 = no limit).  Host-side
 * polling of CUDA events; no device-side wait is involved.  Then reads the
 * workspace status word: a bounded device-side wait that gave up in an
 * attention kernel since the last kvs_sync returns KVS_ERR_CUDA (and clears
 * the word).  Failures are error returns, not aborts (PR "port adaptive KV
 * streaming", review comments); the pages describe no call of this shape. */
kvs_status kvs_sync(kvs_ctx *ctx, uint32_t timeout_ms);

/* kvs_flush -- publish the partial tail page of `layer` (or of every layer if
 * layer == UINT32_MAX) to the host history, e.g. before saving it (the KV
 * writer publishes a changed tail to host: V2 README, "KV data movement and
 * attention"; full pages are published by kvs_append itself). */
kvs_status kvs_flush(kvs_ctx *ctx, uint32_t layer);

/*
 * kvs_page_location -- where page `page` of `layer` is device-readable now:
 * *kind = 0 host only, 1 tail slot, 2 resident pool, 3 leased ring slot
 * (kvs_lease_acquire); *slot = device slot id
 * (or -1).  kvs_read_slot copies device slot `slot` (page_bytes) to host_dst
 * synchronously; kvs_read_host_page copies the host history page.  Debug and
 * test helpers for bit-exact layout and indexing checks; library API with no
 * counterpart on the pages.
 */
kvs_status kvs_page_location(const kvs_ctx *ctx, uint32_t layer, uint64_t page, int32_t *kind,
                             int64_t *slot);
kvs_status kvs_read_slot(kvs_ctx *ctx, int64_t slot, void *host_dst);
kvs_status kvs_read_host_page(kvs_ctx *ctx, uint32_t layer, uint64_t page, void *host_dst);

/* kvs_ring_info -- first device slot id of the ring and its size.  Library
 * API (test helper); no counterpart on the pages. */
kvs_status kvs_ring_info(const kvs_ctx *ctx, int64_t *first_slot, uint32_t *n_slots);

/* kvs_stats -- counters since create (or the last reset when reset != 0).
 * They include the feedback the pages' policy samples (V2 README, "KV data
 * movement and attention": readiness misses, ring occupancy, copy-stream
 * time), in the form kvs_policy_observation takes. */
kvs_status kvs_stats(kvs_ctx *ctx, kvs_stats_t *out, int reset);

/* kvs_set_timing -- library API for measurement (no counterpart on the
 * pages): mask of KVS_TIME_* bits.  Each attention-kernel launch of
 * a selected kind is bracketed by CUDA events on attn_stream; its device time
 * and the page bytes it reads are added to kvs_stats_t.decode_ms /
 * decode_bytes once the events complete.  0 disables. */
#define KVS_TIME_RESIDENT 1u /* launches over tail and resident-pool pages */
#define KVS_TIME_RING 2u     /* launches over ring chunks */
kvs_status kvs_set_timing(kvs_ctx *ctx, int mask);

/*
 * Launch timeline -- library API for measurement (no counterpart on the
 * pages; it shows what the V2 README, "KV data movement and attention",
 * describes: refills for upcoming layers running while the current layer is
 * attended).  Between kvs_timeline_begin and kvs_timeline_end every kernel
 * the context launches takes the next of `max_records` records in the
 * caller's device buffer `records_dev` (16 bytes each, 8-byte aligned): the
 * kernel's first CTA start (stored complemented) and its last CTA end, in
 * %globaltimer nanoseconds, each written by atomic max.  The caller zeroes
 * the records before the launches run (cudaMemsetAsync on attn_stream) --
 * also before each replay of a step graph captured inside the window, whose
 * launches keep the records they were captured with.  Copy-engine refills
 * (KVS_FLAG_DMA_FILL) are not kernels and take no record.  Launches beyond
 * max_records are counted in kvs_timeline_read's *n_dropped and not stamped.
 * kvs_timeline_read (after kvs_sync) copies the records back and returns, per
 * launch, its kind, layer, stream and pages with the two times (0 when the
 * launch has not run).  A new kvs_timeline_begin restarts at record 0.
 */
#define KVS_TL_APPEND 1u      /* quantise rows into the tail page (kvs_append) */
#define KVS_TL_CLEAR 2u       /* zero the tail page's unused token slots */
#define KVS_TL_QPREP 3u       /* query fragments (kvs_attend) */
#define KVS_TL_READ_RESIDENT 4u /* attention over tail and resident-pool pages */
#define KVS_TL_READ_RING 5u   /* attention over one ring chunk */
#define KVS_TL_COMBINE 6u     /* log-sum-exp combine (kvs_attend) */
#define KVS_TL_FILL 7u        /* ring refill: host pages into ring slots */
#define KVS_TL_POOL_LOAD 8u   /* host pages into the resident pool (kvs_set_residency) */
#define KVS_TL_PREFILL 9u     /* tensor-core prefill over one batch of splits */
typedef struct {
    uint32_t kind;      /* KVS_TL_* */
    uint32_t layer;
    int32_t stream;     /* 0 attn_stream, 1 copy_stream, 2k / 2k + 1 lane k's attention /
                           copy stream, 2 n_lanes the resident-page stream, 2 n_lanes + 1
                           lane 0's ring-read stream */
    uint32_t pages;     /* pages the launch reads or moves (0 for other kinds) */
    uint64_t start_ns;  /* first CTA start, %globaltimer */
    uint64_t end_ns;    /* last CTA end */
} kvs_timeline_record;
kvs_status kvs_timeline_begin(kvs_ctx *ctx, void *records_dev, uint32_t max_records);
kvs_status kvs_timeline_end(kvs_ctx *ctx);
kvs_status kvs_timeline_read(kvs_ctx *ctx, kvs_timeline_record *out, uint32_t max_out, uint32_t *n_out,
                             uint32_t *n_dropped);

/*
 * Step graphs.  One decode (or verify) step issues many small launches and
 * ready/consumed handshakes; capturing the step once as a CUDA graph and
 * replaying it removes the host cost of issuing them.  kvs_graph_begin starts
 * stream capture on attn_stream (the copy stream joins it); every kvs_* call
 * until kvs_graph_end is recorded, not executed (host-side state still
 * advances as if it ran once).  No prefetch may be pending at either end.
 * kvs_graph_launch replays the step on attn_stream after the copy stream's
 * earlier work and before its later work; a replay repeats exactly the
 * captured positions, so a captured step should leave the lengths where it
 * found them (e.g. append, attend, truncate).  Replays reuse the device
 * buffers (q, k, v, out, lse) whose addresses were captured.  Attention
 * timing (kvs_set_timing) is not recorded inside a capture.  kvs_set_residency
 * and kvs_set_ring_slots drop a captured graph (its slot schedule is baked in).
 * A graph from an old layout is never reused (V2 README, "Backend-neutral
 * memory and streaming contracts": captured graphs are invalidated at a layout
 * change); the pages' step itself is host-issued, so this API has no direct
 * counterpart there.
 */
kvs_status kvs_graph_begin(kvs_ctx *ctx);
kvs_status kvs_graph_end(kvs_ctx *ctx);
kvs_status kvs_graph_launch(kvs_ctx *ctx);
kvs_status kvs_graph_destroy(kvs_ctx *ctx);

/* kvs_last_error -- library API (no counterpart on the pages): message of the
 * last failed call on ctx ("" if none);
 * with ctx == NULL, the last failure of this thread in a call that takes no
 * context (kvs_query_sizes, kvs_create, kvs_attend_pages_noalloc). */
const char *kvs_last_error(const kvs_ctx *ctx);

/* kvs_debug_inject -- arm a fault (KVS_FAULT_*) that fires on the nth
 * (1-based) matching event; nth = 0 disarms.  Every fault is made on the host
 * or as a shortened device-side wait limit: no GPU fault is ever made.  Test
 * API; the pages describe no such call. */
kvs_status kvs_debug_inject(kvs_ctx *ctx, uint32_t fault, uint64_t nth);

/* kvs_trace_read -- test API (no counterpart on the pages) for checking the
 * span plan's coverage and fences (V2 README, "Backend-neutral memory and
 * streaming contracts": a plan with gaps, overlaps or too little coverage is
 * rejected): copy up to max logged operations of a PLAN_ONLY context
 * starting at index `first` into ops; *n_out = number copied, *n_total = log
 * length.  KVS_ERR_STATE for a context that is not PLAN_ONLY. */
kvs_status kvs_trace_read(const kvs_ctx *ctx, uint64_t first, uint64_t max, kvs_trace_op *ops,
                          uint64_t *n_out, uint64_t *n_total);

/* kvs_version -- KVS_ABI_VERSION of the loaded library (library API; the
 * pages' copy-ops table is versioned the same way: V2 README, "Logical KV
 * layout, policy, and physical execution"). */
int32_t kvs_version(void);

/*
 * kvs_attend_pages_noalloc -- kvs_attend for callers that cannot allocate
 * device memory.  (The pages describe no such call; it exists for callers
 * running inside an allocator or memory-pool callback, plug-ins given a fixed
 * device budget by their host, or services that must not grow their device
 * footprint once running -- none of which can hand kvs_attend a workspace.)
 *
 * Computes the same causal attention as kvs_attend, with no context: the
 * caller passes its pages in one device buffer (pages_dev, pages_bytes) laid
 * out as kvs_query_sizes describes (page_bytes = n_kv_head * page_tokens *
 * head_dim * 13 / 8), a host array page_slots[n_pages] giving the slot of
 * logical page i in that buffer, the queries q_dev [n_rows][n_q_head][D]
 * (KVS_F32 or KVS_F16; row r at position pos0 + r sees keys 0 .. pos0 + r),
 * and outputs out_dev [n_rows][n_q_head][D] fp32 and lse_dev [n_rows][n_q_head]
 * (nullable), all on `stream` (a cudaStream_t).
 * It allocates nothing: split partials go to a fixed 32 MiB device array
 * inside this library, present on every GPU that loads it until the process
 * exits.  A call needing more, i.e. ceil((pos0 + n_rows) / page_tokens) *
 * n_q_head * n_rows * (head_dim + 2) * 4 bytes > 32 MiB, is refused with
 * KVS_ERR_CAPACITY before any work.  The first call on each device looks up
 * the array's device address (cudaGetSymbolAddress); make that first call
 * before any stream capture on that device.  All calls on a device share the
 * array, which keeps the last call's contents: each call first clears the
 * array's timeout flag on `stream` (cudaMemsetAsync, no allocation), and the
 * partials are written before they are read.  Calls whose GPU work overlaps
 * race, so order them on one stream.  A bounded device-side wait that gives
 * up (a copy into shared memory that never completes) cannot be returned as
 * a status, since the call returns before its kernels run: it makes every
 * element of out_dev and lse_dev NaN instead.  pos0 + n_rows beyond INT64_MAX
 * -> KVS_ERR_INVALID.  Works on any device of the process (the scratch address
 * and launch limits are kept per device).  Errors: kvs_last_error(NULL).
 */
kvs_status kvs_attend_pages_noalloc(const void *pages_dev, uint64_t pages_bytes,
                                    const uint32_t *page_slots, uint64_t n_pages,
                                    uint32_t page_tokens, uint32_t n_kv_head, uint32_t head_dim,
                                    const void *q_dev, int32_t q_dtype, uint32_t n_rows,
                                    uint32_t n_q_head, uint64_t pos0, float scale, float *out_dev,
                                    float *lse_dev, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KVS_H_ */
