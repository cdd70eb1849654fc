// kvs host runtime: geometry, host history, page table, resident pool, the
// shared transfer ring with its ready/consumed fences, the span plan and the
// C ABI of include/kvs.h.
//
// Design source: "Adaptive KV Streaming for llama.cpp V2" --
//   "KV data movement and attention": host memory keeps every layer's full
//     history; on the device there are resident pages and a single ring
//     that all layers share; refills for upcoming layers run on a copy
//     stream during the current layer's attention; one event orders a read
//     after its copy, another orders a refill after the last read of the
//     slot; the device budget is the resident pages plus the ring slots.
//   "Keep the stock attention order": one ordered history, resident pages
//     and ring spans (at most two per wrap), then one final reduction.
//   "Backend-neutral memory and streaming contracts": the span plan covers
//     the history without gaps or overlaps.
// and "Adaptive KV Streaming for llama.cpp", "Adaptive KV streaming":
//   a ring slot is reused as soon as its last read has run.
//
// Scheduling model.  Nonresident pages are grouped, layer by layer in the
// order layers are announced, into chunks of up to chunk_pages pages.  Each
// page of the global chunk sequence takes the next ring sequence number and
// lives in slot seq % ring_slots.  A chunk's copy is enqueued only when the
// attention of every chunk that last used its slots has been enqueued; the
// copy waits on the newest of those chunks' consumed events (attention is
// in order, so that implies the older ones), copies, and records its own
// ready event.  Attention waits on ready, reads, and records consumed.  Each
// chunk holds at least one slot, so at most ring_slots chunks are live and
// ring_slots ready/consumed events, indexed by chunk id, suffice.
#include <cuda_runtime.h>
#include <stddef.h>
#include <string.h>

#include <algorithm>
#include <climits>
#include <chrono>
#include <deque>
#include <string>
#include <thread>
#include <vector>

#include "kvs.h"
#include "kvs_internal.h"

using kvs::PageGeom;

namespace {

thread_local std::string g_create_error;

constexpr int kAttn = 0;
constexpr int kCopy = 1;

struct Chunk {
    uint64_t id;
    uint32_t layer;
    uint64_t seq0;               // ring sequence number of its first page
    std::vector<int64_t> pages;  // logical pages, ascending
    bool filled = false;
};

struct Timer {
    cudaEvent_t start, stop;
    uint64_t bytes;
};

struct LayerState {
    uint64_t T = 0;                  // tokens appended
    std::vector<uint8_t> mask;       // requested residency per page
    std::vector<int64_t> pool_slot;  // pool slot per page or -1
    int64_t tail_page[2] = {-1, -1};  // page held by tail slot (page % 2)
};

}  // namespace

struct kvs_ctx {
    kvs_config cfg;
    PageGeom geom;
    bool plan_only = false;
    cudaStream_t attn = nullptr, copy = nullptr;  // lane 0
    int n_lanes = 1;
    std::vector<cudaStream_t> lanes;  // stream id s: lane s/2, attention if s even, copy if odd
    std::string err;

    // device page slots: [0, 2L) tails, [2L, 2L + pool_n) pool, then the ring
    int64_t n_slots = 0, pool_n = 0, ring_first = 0;
    uint32_t ring_n = 0, chunk_pages = 1;
    std::vector<int32_t> pool_layer;  // owner layer per pool slot (-1 free)
    std::vector<int64_t> pool_page;
    int64_t pool_used = 0;

    int64_t max_pages = 0;
    int64_t prefill_split = 24;  // pages per tensor-core prefill split
    bool split_chunks = false;  // ring chunks stop at prefill split boundaries (prefill-capable context)
    uint32_t verify_rows = 1;   // widest split-K call (row groups beyond 64 rows x heads)
    // complete-layer lease: slots [ring_first + ring_n, ring_first + lease_ring_full)
    // are taken out of the ring and hold the leased layer's nonresident pages
    kvs_policy_observation last_obs = {};  // the last kvs_observe result
    int64_t lease_layer = -1;
    uint32_t lease_ring_full = 0;       // ring size before the lease
    std::vector<int64_t> lease_spare;   // leased slots not holding a page yet
    int64_t qfrag_groups = 1;   // query-fragment areas in the workspace (one per row group)
    bool check_status = false;  // a kernel with bounded device waits ran since the last kvs_sync
    std::vector<LayerState> layers;

    uint8_t *host = nullptr;      // host history (host address)
    uint8_t *host_dev = nullptr;  // same bytes, device-visible address
    bool host_registered = false;

    // ring scheduler
    uint64_t ring_seq = 0, next_chunk = 0, attended = 0;
    std::vector<int64_t> slot_last_chunk;  // per ring slot, -1 if never used
    std::deque<Chunk> queue;               // planned chunks, not yet attended
    std::deque<uint32_t> announced;        // layers announced by prefetch/attend, in order

    // events: [0, R) ready, [R, 2R) consumed, 2R attn mark, 2R+1 copy mark,
    // one publish event per tail slot, then one mark per lane stream
    std::vector<cudaEvent_t> events;
    int ev_attn_mark = 0, ev_copy_mark = 0, ev_pub0 = 0, ev_lane0 = 0, ev_pub_last = 0, ev_clear0 = 0;
    // per layer: a truncate's tail clear is queued on the resident-page stream and
    // the attention stream has not waited for it yet (settle_clear)
    std::vector<uint8_t> clear_pending;
    uint64_t pub_generation = 0;        // publishes recorded on the copy stream
    std::vector<uint64_t> lane_pub_seen;  // per stream: pub_generation it has waited for
    std::vector<uint64_t> page_pub_gen;   // per (layer, page): pub_generation of its last publish
    std::vector<int> chunk_reader_sid;    // per chunk id % ring_n: stream its attention read ran on

    // timing of attention kernels (mask of KVS_TIME_*)
    uint32_t timing = 0;
    std::vector<cudaEvent_t> timer_free;
    std::vector<Timer> timer_pending;

    // step graph capture / replay
    bool capturing = false;
    std::vector<uint8_t> ev_in_capture;  // event recorded since capture began
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t graph_exec = nullptr;
    std::vector<cudaEvent_t> eager_events;  // the context's events while a capture is open
    std::vector<cudaEvent_t> graph_events;  // events owned by the captured graph
    uint64_t graph_kernel_base = 0, graph_kernels = 0;

    // fault injection
    uint32_t fault = KVS_FAULT_NONE;
    uint64_t fault_nth = 0, fault_count = 0;

    kvs_stats_t st;
    std::vector<kvs_trace_op> trace;

    int64_t tail_slot(uint32_t layer, int64_t page) const { return 2 * (int64_t)layer + (page & 1); }
    int64_t pool_slot_id(int64_t i) const { return 2 * (int64_t)cfg.n_layers + i; }
    int64_t ring_slot_id(uint64_t seq) const { return ring_first + (int64_t)(seq % ring_n); }
    uint8_t *slot_ptr(int64_t slot) const {
        return static_cast<uint8_t *>(cfg.arena) + slot * geom.page_bytes;
    }
    uint8_t *host_page(uint32_t layer, int64_t page) const {
        return host + ((int64_t)layer * max_pages + page) * geom.page_bytes;
    }
    uint8_t *host_page_dev(uint32_t layer, int64_t page) const {
        return host_dev + ((int64_t)layer * max_pages + page) * geom.page_bytes;
    }
    cudaStream_t stream(int s) const { return lanes[s]; }
    // lane streams, then the library's own resident-page stream (res_sid()) and
    // the stream that reads lane 0's ring chunks (ring0_sid()), so that the
    // caller's attention stream carries only the per-call work (Q prep, the
    // combine, appends) and never waits behind ring refills
    int n_streams() const { return 2 * n_lanes + 2; }
    int res_sid() const { return 2 * n_lanes; }
    int ring0_sid() const { return 2 * n_lanes + 1; }
    int attn_sid_of_lane(int lane) const { return lane == 0 ? ring0_sid() : 2 * lane; }
    // launch timeline (kvs_timeline_begin): the caller's device records and per-record meta
    unsigned long long *tl_buf = nullptr;
    uint32_t tl_max = 0, tl_dropped = 0;
    bool tl_on = false;
    std::vector<kvs_timeline_record> tl_meta;
    cudaStream_t res_stream = nullptr;    // created by kvs_create, lowest priority
    cudaStream_t ring0_stream = nullptr;  // created by kvs_create
    ~kvs_ctx() {
        if (res_stream) cudaStreamDestroy(res_stream);
        if (ring0_stream) cudaStreamDestroy(ring0_stream);
    }
};

namespace {

kvs_status fail(kvs_ctx *c, kvs_status s, const std::string &msg) {
    if (c) c->err = msg;
    return s;
}

kvs_status cuda_fail(kvs_ctx *c, cudaError_t e, const char *what) {
    return fail(c, KVS_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

void log_op(kvs_ctx *c, uint32_t op, int stream, uint32_t layer, uint32_t ev, int64_t a, int64_t b,
            int64_t cc = 0) {
    kvs_trace_op t;
    t.op = op;
    t.stream = (uint32_t)stream;
    t.layer = layer;
    t.event = ev;
    t.a = a;
    t.b = b;
    t.c = cc;
    t.d = 0;
    c->trace.push_back(t);
}

// ---- stream primitives (logged in plan-only mode, executed otherwise)

kvs_status op_record(kvs_ctx *c, int stream, int ev) {
    if (c->capturing) c->ev_in_capture[ev] = 1;
    if (c->plan_only) {
        log_op(c, KVS_OP_RECORD, stream, 0, (uint32_t)ev, 0, 0);
        return KVS_OK;
    }
    cudaError_t e = cudaEventRecord(c->events[ev], c->stream(stream));
    return e == cudaSuccess ? KVS_OK : cuda_fail(c, e, "cudaEventRecord");
}

kvs_status op_wait(kvs_ctx *c, int stream, int ev) {
    // inside a step graph, an event last recorded before capture began was
    // already covered by the join kvs_graph_launch makes before each replay
    if (c->capturing && !c->ev_in_capture[ev]) return KVS_OK;
    if (c->plan_only) {
        log_op(c, KVS_OP_WAIT, stream, 0, (uint32_t)ev, 0, 0);
        return KVS_OK;
    }
    cudaError_t e = cudaStreamWaitEvent(c->stream(stream), c->events[ev], 0);
    return e == cudaSuccess ? KVS_OK : cuda_fail(c, e, "cudaStreamWaitEvent");
}

// attention stream waits for everything enqueued so far on the copy stream
kvs_status join_copy_into_attn(kvs_ctx *c) {
    kvs_status s = op_record(c, kCopy, c->ev_copy_mark);
    return s != KVS_OK ? s : op_wait(c, kAttn, c->ev_copy_mark);
}

// copy stream waits for everything enqueued so far on the attention stream
kvs_status join_attn_into_copy(kvs_ctx *c) {
    kvs_status s = op_record(c, kAttn, c->ev_attn_mark);
    return s != KVS_OK ? s : op_wait(c, kCopy, c->ev_attn_mark);
}

// stream `to` waits for everything enqueued so far on stream `from`
kvs_status join(kvs_ctx *c, int from, int to) {
    kvs_status s = op_record(c, from, c->ev_lane0 + from);
    return s != KVS_OK ? s : op_wait(c, to, c->ev_lane0 + from);
}

// every other lane stream waits for the primary stream of its kind (the
// resident-page stream counts as an attention stream)
kvs_status fork_lanes(kvs_ctx *c) {
    for (int l = 1; l < c->n_lanes; ++l) {
        kvs_status s = join(c, kAttn, 2 * l);
        if (s == KVS_OK) s = join(c, kCopy, 2 * l + 1);
        if (s != KVS_OK) return s;
    }
    kvs_status s = join(c, kAttn, c->res_sid());
    return s != KVS_OK ? s : join(c, kAttn, c->ring0_sid());
}

// the other attention streams wait for the primary attention stream (inputs
// of this call in place, the previous combine done with the partials)
kvs_status fork_attn_lanes(kvs_ctx *c) {
    for (int l = 1; l < c->n_lanes; ++l) {
        kvs_status s = join(c, kAttn, 2 * l);
        if (s != KVS_OK) return s;
    }
    kvs_status s = join(c, kAttn, c->res_sid());
    return s != KVS_OK ? s : join(c, kAttn, c->ring0_sid());
}

// a publish (D2H of a completed tail page) was just enqueued on the copy
// stream: a copy lane that later refills that page from host waits for it once
kvs_status mark_publish(kvs_ctx *c, uint32_t layer, int64_t page) {
    kvs_status s = op_record(c, kCopy, c->ev_pub_last);
    if (s == KVS_OK) c->pub_generation++;
    c->page_pub_gen[(size_t)layer * (size_t)c->max_pages + (size_t)page] = c->pub_generation;
    c->lane_pub_seen[kCopy] = c->pub_generation;  // the copy stream itself
    return s;
}

// the primary attention stream waits for the other attention streams
kvs_status join_attn_lanes_into_attn(kvs_ctx *c) {
    for (int sid = 2; sid <= c->res_sid(); sid += 2) {
        kvs_status s = join(c, sid, kAttn);
        if (s != KVS_OK) return s;
    }
    return join(c, c->ring0_sid(), kAttn);
}

// the primary attention stream waits for every other stream of every lane
kvs_status join_all_into_attn(kvs_ctx *c) {
    for (int sid = 1; sid < c->n_streams(); ++sid) {
        kvs_status s = join(c, sid, kAttn);
        if (s != KVS_OK) return s;
    }
    std::fill(c->clear_pending.begin(), c->clear_pending.end(), 0);  // the resident-page stream joined
    return KVS_OK;
}

// A truncate zeroes the dropped token slots of the tail page on the
// resident-page stream, so the clear is not a link of the attention stream's
// layer-to-layer chain.  Work on the attention stream that touches that
// layer's tail slots waits for it first (everything ordered after the
// attention stream then is too); resident reads on the resident-page stream
// follow it in stream order.
kvs_status settle_clear(kvs_ctx *c, uint32_t layer) {
    if (layer >= c->clear_pending.size() || !c->clear_pending[layer]) return KVS_OK;
    kvs_status s = op_wait(c, kAttn, c->ev_clear0 + (int)layer);
    if (s == KVS_OK) c->clear_pending[layer] = 0;
    return s;
}

kvs_status settle_clears(kvs_ctx *c, uint32_t l0, uint32_t l1) {
    for (uint32_t l = l0; l < l1 && l < c->clear_pending.size(); ++l) {
        kvs_status s = settle_clear(c, l);
        if (s != KVS_OK) return s;
    }
    return KVS_OK;
}

// the next timeline record for a launch (null when the timeline is off or full)
unsigned long long *tl_take(kvs_ctx *c, uint32_t kind, uint32_t layer, int sid, uint32_t pages = 0) {
    if (!c->tl_on || c->plan_only) return nullptr;
    if (c->tl_meta.size() >= c->tl_max) {
        c->tl_dropped++;
        return nullptr;
    }
    kvs_timeline_record r = {};
    r.kind = kind;
    r.layer = layer;
    r.stream = sid;
    r.pages = pages;
    c->tl_meta.push_back(r);
    return c->tl_buf + 2 * (c->tl_meta.size() - 1);
}

// host pages -> device slots on the copy stream (ring fill or pool load)
// observation record of ring chunk `id` in the workspace (null in plan-only mode)
unsigned long long *obs_record(kvs_ctx *c, uint64_t id);
unsigned long long *obs_accumulator(kvs_ctx *c);

kvs_status op_copy_pages(kvs_ctx *c, uint32_t layer, const std::vector<int64_t> &pages,
                         const std::vector<int64_t> &slots, uint32_t kind,
                         const std::vector<uint64_t> *seqs, int sid = kCopy, bool pdl = false,
                         unsigned long long *rec = nullptr) {
    if (!(c->cfg.flags & KVS_FLAG_DMA_FILL))
        c->st.kernel_launches += (pages.size() + kvs::kMaxFillPages - 1) / kvs::kMaxFillPages;
    if (c->plan_only) {
        for (size_t i = 0; i < pages.size(); ++i)
            log_op(c, kind, sid, layer, 0, pages[i], slots[i], seqs ? (int64_t)(*seqs)[i] : 0);
        return KVS_OK;
    }
    if (c->cfg.flags & KVS_FLAG_DMA_FILL) {
        for (size_t i = 0; i < pages.size();) {
            size_t j = i + 1;
            while (j < pages.size() && pages[j] == pages[j - 1] + 1 && slots[j] == slots[j - 1] + 1) ++j;
            cudaError_t e = cudaMemcpyAsync(c->slot_ptr(slots[i]), c->host_page(layer, pages[i]),
                                            (size_t)(j - i) * (size_t)c->geom.page_bytes, cudaMemcpyHostToDevice,
                                            c->stream(sid));
            if (e != cudaSuccess) return cuda_fail(c, e, "ring/pool copy");
            i = j;
        }
        return KVS_OK;
    }
    for (size_t i0 = 0; i0 < pages.size(); i0 += kvs::kMaxFillPages) {
        kvs::FillParams fp;
        fp.rec = rec;
        fp.n = (int)std::min<size_t>(kvs::kMaxFillPages, pages.size() - i0);
        fp.tl = tl_take(c, kind == KVS_OP_FILL ? KVS_TL_FILL : KVS_TL_POOL_LOAD, layer, sid, (uint32_t)fp.n);
        fp.page_bytes = c->geom.page_bytes;
        for (int j = 0; j < fp.n; ++j) {
            fp.src[j] = c->host_page_dev(layer, pages[i0 + j]);
            fp.dst[j] = c->slot_ptr(slots[i0 + j]);
        }
        cudaError_t e = kvs::launch_fill(fp, c->stream(sid), pdl && i0 == 0);
        if (e != cudaSuccess) return cuda_fail(c, e, "ring/pool fill launch");
    }
    return KVS_OK;
}

kvs_status take_timer_event(kvs_ctx *c, cudaEvent_t *ev) {
    if (c->timer_free.empty()) {
        cudaEvent_t e;
        cudaError_t r = cudaEventCreate(&e);
        if (r != cudaSuccess) return cuda_fail(c, r, "cudaEventCreate");
        c->timer_free.push_back(e);
    }
    *ev = c->timer_free.back();
    c->timer_free.pop_back();
    return KVS_OK;
}

kvs_status timed_begin(kvs_ctx *c, uint32_t kind, cudaEvent_t *ev, int sid) {
    *ev = nullptr;
    // graph-recorded events carry no timing: no timers inside a step capture
    if (!(c->timing & kind) || c->plan_only || c->capturing) return KVS_OK;
    kvs_status s = take_timer_event(c, ev);
    if (s != KVS_OK) return s;
    cudaError_t r = cudaEventRecord(*ev, c->stream(sid));
    return r == cudaSuccess ? KVS_OK : cuda_fail(c, r, "cudaEventRecord");
}

kvs_status timed_end(kvs_ctx *c, cudaEvent_t start, uint64_t bytes, int sid) {
    if (!start) return KVS_OK;
    cudaEvent_t stop = nullptr;
    kvs_status s = take_timer_event(c, &stop);
    if (s != KVS_OK) return s;
    cudaError_t r = cudaEventRecord(stop, c->stream(sid));
    if (r != cudaSuccess) return cuda_fail(c, r, "cudaEventRecord");
    c->timer_pending.push_back({start, stop, bytes});
    return KVS_OK;
}

void harvest_timers(kvs_ctx *c) {
    std::vector<Timer> keep;
    for (auto &t : c->timer_pending) {
        if (cudaEventQuery(t.stop) == cudaSuccess) {
            float ms = 0.f;
            if (cudaEventElapsedTime(&ms, t.start, t.stop) == cudaSuccess) {
                c->st.decode_ms += ms;
                c->st.decode_timed += 1;
                c->st.decode_bytes += t.bytes;
            }
            c->timer_free.push_back(t.start);
            c->timer_free.push_back(t.stop);
        } else {
            keep.push_back(t);
        }
    }
    c->timer_pending.swap(keep);
}

// ---- events

void destroy_events(kvs_ctx *c) {
    if (!c->plan_only)
        for (cudaEvent_t e : c->events)
            if (e) cudaEventDestroy(e);
    c->events.clear();
}

kvs_status create_events(kvs_ctx *c) {
    const int R = (int)c->ring_n;
    const int n = 2 * R + 2 + 2 * (int)c->cfg.n_layers + c->n_streams() + 1 + (int)c->cfg.n_layers;
    c->ev_attn_mark = 2 * R;
    c->ev_copy_mark = 2 * R + 1;
    c->ev_pub0 = 2 * R + 2;
    c->ev_lane0 = c->ev_pub0 + 2 * (int)c->cfg.n_layers;
    c->ev_pub_last = c->ev_lane0 + c->n_streams();
    c->ev_clear0 = c->ev_pub_last + 1;
    c->clear_pending.assign(c->cfg.n_layers, 0);
    c->pub_generation = 0;
    c->lane_pub_seen.assign(c->n_streams(), 0);
    c->events.assign(n, nullptr);
    if (c->plan_only) return KVS_OK;
    for (int i = 0; i < n; ++i) {
        cudaError_t e = cudaEventCreateWithFlags(&c->events[i], cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(c, e, "cudaEventCreate");
    }
    return KVS_OK;
}

void release_graph(kvs_ctx *c) {
    if (c->plan_only) return;
    if (c->graph_exec) cudaGraphExecDestroy(c->graph_exec);
    if (c->graph) cudaGraphDestroy(c->graph);
    for (cudaEvent_t e : c->graph_events)
        if (e) cudaEventDestroy(e);
    c->graph_exec = nullptr;
    c->graph = nullptr;
    c->graph_events.clear();
}

// ---- placement

// 1: tail slot, 2: pool, 0: host only
int locate(const kvs_ctx *c, uint32_t layer, int64_t page, int64_t *slot) {
    const LayerState &L = c->layers[layer];
    if (L.tail_page[page & 1] == page) {
        *slot = c->tail_slot(layer, page);
        return 1;
    }
    if (page < (int64_t)L.pool_slot.size() && L.pool_slot[page] >= 0) {
        *slot = L.pool_slot[page];
        return 2;
    }
    *slot = -1;
    return 0;
}

int64_t n_pages_of(const kvs_ctx *c, uint32_t layer) {
    return (int64_t)((c->layers[layer].T + c->geom.P - 1) / c->geom.P);
}

int64_t pool_alloc(kvs_ctx *c, uint32_t layer, int64_t page) {
    for (int64_t i = 0; i < c->pool_n; ++i) {
        if (c->pool_layer[i] < 0) {
            c->pool_layer[i] = (int32_t)layer;
            c->pool_page[i] = page;
            c->pool_used++;
            return c->pool_slot_id(i);
        }
    }
    return -1;
}

void pool_free(kvs_ctx *c, int64_t slot) {
    const int64_t i = slot - 2 * (int64_t)c->cfg.n_layers;
    if (i >= 0 && i < c->pool_n && c->pool_layer[i] >= 0) {
        c->pool_layer[i] = -1;
        c->pool_page[i] = -1;
        c->pool_used--;
    }
}

bool is_lease_slot(const kvs_ctx *c, int64_t slot) {
    return c->lease_layer >= 0 && slot >= c->ring_first + (int64_t)c->ring_n &&
           slot < c->ring_first + (int64_t)c->lease_ring_full;
}

bool layer_has_plan(const kvs_ctx *c, uint32_t layer) {
    return std::find(c->announced.begin(), c->announced.end(), layer) != c->announced.end();
}

// Where a page leaving its tail slot goes: 1 = resident pool, 0 = host only
// (streamed later), 2 = host only and appended to the layer's pending plan,
// -1 = nowhere (pending plan not last in the queue and no free pool slot).
int evict_target(const kvs_ctx *c, uint32_t layer, int64_t page, int64_t free_pool) {
    const LayerState &L = c->layers[layer];
    const bool want = page < (int64_t)L.mask.size() && L.mask[page];
    const bool planned = layer_has_plan(c, layer);
    if (want && free_pool > 0) return 1;
    if (!planned) return 0;
    if (c->announced.back() == layer) return 2;
    return free_pool > 0 ? 1 : -1;
}

// ---- ring scheduling

// chunk size when the caller leaves it open: a quarter of the ring, so four
// chunks are in flight, and at most 32 pages so one chunk's copy stays short
uint32_t default_chunk_pages(uint32_t ring_slots) {
    return std::min(32u, std::max(1u, ring_slots / 4));
}

// Plan the nonresident pages of `layer` into chunks at the end of the queue.
void plan_layer(kvs_ctx *c, uint32_t layer) {
    const int64_t np = n_pages_of(c, layer);
    std::vector<int64_t> streamed;
    for (int64_t p = 0; p < np; ++p) {
        int64_t s;
        if (locate(c, layer, p, &s) == 0) streamed.push_back(p);
    }
    // chunks of up to chunk_pages pages; in a context that can run the prefill
    // path they never cross a prefill split (that path attends split by split)
    const int64_t align = c->split_chunks ? c->prefill_split : INT64_MAX;
    for (size_t i = 0; i < streamed.size();) {
        Chunk ch;
        ch.id = c->next_chunk++;
        ch.layer = layer;
        ch.seq0 = c->ring_seq;
        const int64_t split = streamed[i] / align;
        size_t n = 0;
        while (i + n < streamed.size() && n < c->chunk_pages && streamed[i + n] / align == split) ++n;
        ch.pages.assign(streamed.begin() + i, streamed.begin() + i + n);
        c->ring_seq += n;
        i += n;
        c->queue.push_back(std::move(ch));
    }
    c->announced.push_back(layer);
}

bool fill_possible(const kvs_ctx *c, const Chunk &ch) {
    for (size_t i = 0; i < ch.pages.size(); ++i) {
        const int64_t prev = c->slot_last_chunk[(ch.seq0 + i) % c->ring_n];
        if (prev >= 0 && (uint64_t)prev >= c->attended) return false;
    }
    return true;
}

kvs_status fill_chunk(kvs_ctx *c, Chunk &ch) {
    if (c->fault == KVS_FAULT_FILL_ENQUEUE && c->fault_nth) {
        if (++c->fault_count == c->fault_nth)
            return fail(c, KVS_ERR_INJECTED, "injected fault: ring refill enqueue");
    }
    // the last reader of every slot (readers may sit on different streams)
    std::vector<int64_t> prev;
    for (size_t i = 0; i < ch.pages.size(); ++i) {
        const int64_t p = c->slot_last_chunk[(ch.seq0 + i) % c->ring_n];
        if (p >= 0 && std::find(prev.begin(), prev.end(), p) == prev.end()) prev.push_back(p);
    }
    // Immediate recycle: when every previous reader ran on one attention
    // stream, the refill follows them on that stream as a programmatic
    // dependent launch.  An attention CTA signals its dependents once its
    // page sections sit in shared memory, so the copy overlaps the rest of
    // the read; stream order covers the slots.  Otherwise the refill goes to
    // the chunk's copy lane and waits for each reader's consumed event.
    int sid = 2 * (int)(ch.id % (uint64_t)c->n_lanes) + 1;  // this chunk's copy lane
    bool follow = !prev.empty();
    const int rsid = follow ? c->chunk_reader_sid[prev[0] % c->ring_n] : -1;
    for (int64_t p : prev) follow = follow && rsid >= 0 && c->chunk_reader_sid[p % c->ring_n] == rsid;
    // a refill never follows a read on the caller's attention stream, where it
    // would hold up the combine and the next call's work
    if (rsid == kAttn) follow = false;
    kvs_status s;
    if (follow) {
        sid = rsid;
    } else {
        for (int64_t p : prev) {
            s = op_wait(c, sid, (int)c->ring_n + (int)(p % c->ring_n));
            if (s != KVS_OK) return s;
        }
    }
    // a page of this chunk published since this lane last waited: wait for the
    // publishes (the copy stream runs them in order, so the last one covers all)
    uint64_t need = 0;
    for (int64_t p : ch.pages)
        need = std::max(need, c->page_pub_gen[(size_t)ch.layer * (size_t)c->max_pages + (size_t)p]);
    if (c->lane_pub_seen[sid] < need) {
        s = op_wait(c, sid, c->ev_pub_last);
        if (s != KVS_OK) return s;
        c->lane_pub_seen[sid] = c->pub_generation;
    }
    std::vector<int64_t> slots(ch.pages.size());
    std::vector<uint64_t> seqs(ch.pages.size());
    for (size_t i = 0; i < ch.pages.size(); ++i) {
        seqs[i] = ch.seq0 + i;
        slots[i] = c->ring_slot_id(ch.seq0 + i);
    }
    s = op_copy_pages(c, ch.layer, ch.pages, slots, KVS_OP_FILL, &seqs, sid, follow, obs_record(c, ch.id));
    if (s != KVS_OK) return s;
    s = op_record(c, sid, (int)(ch.id % c->ring_n));
    if (s != KVS_OK) return s;
    for (size_t i = 0; i < ch.pages.size(); ++i) {
        int64_t &last = c->slot_last_chunk[(ch.seq0 + i) % c->ring_n];
        if (last >= 0) c->st.ring_recycles++;
        last = (int64_t)ch.id;
    }
    c->chunk_reader_sid[ch.id % c->ring_n] = -1;
    c->st.h2d_pages += ch.pages.size();
    c->st.h2d_bytes += ch.pages.size() * (uint64_t)c->geom.page_bytes;
    c->st.h2d_launches += 1;
    ch.filled = true;
    return KVS_OK;
}

// Enqueue every copy that may go now, in queue order.
kvs_status pump(kvs_ctx *c) {
    for (Chunk &ch : c->queue) {
        if (ch.filled) continue;
        if (!fill_possible(c, ch)) break;
        kvs_status s = fill_chunk(c, ch);
        if (s != KVS_OK) return s;
    }
    return KVS_OK;
}

// ---- attention launches

kvs_status launch_items(kvs_ctx *c, uint32_t layer, const std::vector<int64_t> &pages,
                        const std::vector<int64_t> &slots, kvs::DecodeParams &dp, uint32_t kind,
                        int sid = kAttn) {
    for (size_t i0 = 0; i0 < pages.size(); i0 += kvs::kMaxItems) {
        const int n = (int)std::min<size_t>(kvs::kMaxItems, pages.size() - i0);
        c->st.decode_launches++;
        c->st.kernel_launches++;
        if (c->plan_only) {
            log_op(c, KVS_OP_LAUNCH, sid, layer, 0, 1, n);
            for (int j = 0; j < n; ++j)
                for (int g = 0; g < c->geom.Hk; ++g)
                    log_op(c, KVS_OP_READ, sid, layer, 0, pages[i0 + j], slots[i0 + j], g);
            continue;
        }
        dp.n_items = n;
        // ring chunks: one CTA per (page, kv head, row tile), so the chunk's
        // slots are read (and can be refilled) as soon as possible
        dp.tile_mode = kind == KVS_TIME_RING ? 1 : 0;
        // a small chunk read's signal sits on its refill's path (decode32k: 16 CTAs
        // per read, refills 1.5 us sooner, +1.5%); with large chunks (long262k:
        // 128 CTAs per read) the sooner refills overlapped more and the link ran
        // a few percent slower, so those signal after the softmax
        dp.early_dependents = dp.tile_mode && n * c->geom.Hk * (int)((dp.G * dp.Rg + 7) / 8) <= 64;
        for (int j = 0; j < n; ++j) {
            dp.page[j] = (uint32_t)pages[i0 + j];
            dp.slot[j] = (uint32_t)slots[i0 + j];
        }
        cudaEvent_t t0;
        kvs_status s = timed_begin(c, kind, &t0, sid);
        if (s != KVS_OK) return s;
        if (i0 > 0) dp.rec = nullptr;  // one record per chunk
        dp.tl = tl_take(c, kind == KVS_TIME_RING ? KVS_TL_READ_RING : KVS_TL_READ_RESIDENT, layer, sid, (uint32_t)n);
        cudaError_t e = kvs::launch_decode(dp, c->stream(sid));
        if (e != cudaSuccess) return cuda_fail(c, e, "attention kernel launch");
        c->check_status = true;
        s = timed_end(c, t0, (uint64_t)n * (uint64_t)c->geom.page_bytes, sid);
        if (s != KVS_OK) return s;
    }
    return KVS_OK;
}

// workspace: [status word at 0, observation accumulator at 64 | 256 B]
// [observation records | kObsRecords x 16 B][query fragments][partials]
constexpr uint64_t kStatusBytes = 256;
constexpr uint64_t kAccOffset = 64;
constexpr uint64_t kObsBytes = (uint64_t)kvs::kObsRecords * 16;

unsigned long long *obs_record(kvs_ctx *c, uint64_t id) {
    if (c->plan_only) return nullptr;
    return reinterpret_cast<unsigned long long *>(static_cast<uint8_t *>(c->cfg.workspace) + kStatusBytes) +
           2 * (id % (uint64_t)kvs::kObsRecords);
}
unsigned long long *obs_accumulator(kvs_ctx *c) {
    if (c->plan_only) return nullptr;
    return reinterpret_cast<unsigned long long *>(static_cast<uint8_t *>(c->cfg.workspace) + kAccOffset);
}

// the tensor-core prefill path serves fp16 queries at head_dim 256 with pages
// of a multiple of 64 tokens
bool prefill_geometry(uint32_t D, uint32_t P) { return D == 256 && P % 64 == 0; }

// query rows per split-K row group (its MMA tile holds 64 rows x heads)
uint32_t rows_per_group(uint32_t G) { return std::max<uint32_t>(1, (uint32_t)kvs::decode_max_mma_rows() / G); }

// widest call the split-K kernel serves, as row groups (kvs_config.max_verify_rows)
uint64_t verify_rows_of(const kvs_config *cfg) {
    const uint32_t G = cfg->max_q_head / std::max<uint32_t>(1, cfg->n_kv_head);
    if (cfg->max_verify_rows) return std::min<uint64_t>(cfg->max_verify_rows, cfg->max_rows);
    if (prefill_geometry(cfg->head_dim, cfg->page_tokens)) return std::min<uint64_t>(cfg->max_rows, rows_per_group(G));
    return cfg->max_rows;
}

uint64_t prefill_split_of(const kvs_config *cfg) {
    uint64_t sp = cfg->prefill_split_pages ? cfg->prefill_split_pages : 24;
    sp = std::min<uint64_t>(sp, (uint64_t)kvs::kMaxPrefillSplitPages);
    const uint64_t ring = cfg->ring_slots ? cfg->ring_slots : 1;
    return std::max<uint64_t>(1, std::min(sp, ring));
}

bool geometry_ok(const kvs_config *cfg, std::string *why) {
    const uint32_t P = cfg->page_tokens, D = cfg->head_dim;
    if (!(P == 32 || P == 64 || P == 128 || P == 256)) {
        *why = "page_tokens must be 32, 64, 128 or 256";
        return false;
    }
    if (!(D == 64 || D == 128 || D == 256)) {
        *why = "head_dim must be 64, 128 or 256";
        return false;
    }
    if (cfg->n_kv_head < 1 || cfg->n_layers < 1 || cfg->max_tokens < 1) {
        *why = "n_kv_head, n_layers and max_tokens must be positive";
        return false;
    }
    if (cfg->max_q_head < cfg->n_kv_head || cfg->max_q_head % cfg->n_kv_head != 0) {
        *why = "max_q_head must be a positive multiple of n_kv_head";
        return false;
    }
    if (cfg->max_rows < 1 || cfg->max_rows > 256) {
        *why = "max_rows must be in 1..256";
        return false;
    }
    if (cfg->k_type != KVS_TYPE_Q8_0 || cfg->v_type != KVS_TYPE_Q4_0) {
        *why = "only K = Q8_0 and V = Q4_0 are served";
        return false;
    }
    return true;
}

void sizes_of(const kvs_config *cfg, uint64_t *page_bytes, uint64_t *host_bytes, uint64_t *arena_min,
              uint64_t *ws_min) {
    const PageGeom g = kvs::make_geom((int)cfg->page_tokens, (int)cfg->n_kv_head, (int)cfg->head_dim);
    const uint64_t max_pages = (cfg->max_tokens + cfg->page_tokens - 1) / cfg->page_tokens;
    const uint64_t ring = cfg->ring_slots ? cfg->ring_slots : 1;
    if (page_bytes) *page_bytes = (uint64_t)g.page_bytes;
    if (host_bytes) *host_bytes = (uint64_t)cfg->n_layers * max_pages * (uint64_t)g.page_bytes;
    if (arena_min) *arena_min = (2ull * cfg->n_layers + ring) * (uint64_t)g.page_bytes;
    if (ws_min) {
        // split-K (decode, verify, wide verify as row groups): one partial per page
        // for every (row, head) of a call of up to max_verify_rows rows
        // (any call within 64 rows x heads per kv head, and any row-group call)
        const uint64_t vrows = verify_rows_of(cfg);
        const uint64_t dec_rows = std::max<uint64_t>(
            std::min<uint64_t>((uint64_t)cfg->max_q_head * cfg->max_rows, 64ull * cfg->n_kv_head),
            (uint64_t)cfg->max_q_head * vrows);
        uint64_t need = max_pages * dec_rows * (uint64_t)(cfg->head_dim + 2) * 4ull;
        // prefill: one partial per split
        if ((uint64_t)cfg->max_q_head * cfg->max_rows > 64ull * cfg->n_kv_head &&
            prefill_geometry(cfg->head_dim, cfg->page_tokens)) {
            const uint64_t sp = prefill_split_of(cfg);
            const uint64_t splits = (max_pages + sp - 1) / sp;
            need = std::max<uint64_t>(need, splits * cfg->max_q_head * cfg->max_rows *
                                                (uint64_t)(cfg->head_dim + 2) * 4ull);
        }
        // query fragments of every row group of the widest split-K call
        const uint32_t G = cfg->max_q_head / cfg->n_kv_head;
        const uint64_t groups = (vrows + rows_per_group(G) - 1) / rows_per_group(G);
        *ws_min = kStatusBytes + kObsBytes + groups * (uint64_t)kvs::qfrag_bytes((int)cfg->n_kv_head, (int)cfg->head_dim) +
                  need;
    }
}

}  // namespace

namespace kvs {
void set_thread_error(const std::string &msg) { g_create_error = msg; }
}  // namespace kvs

// ======================================================================= C ABI

extern "C" {

int32_t kvs_version(void) { return KVS_ABI_VERSION; }

const char *kvs_last_error(const kvs_ctx *ctx) {
    return ctx ? ctx->err.c_str() : g_create_error.c_str();
}

kvs_status kvs_query_sizes(const kvs_config *cfg, uint64_t *page_bytes, uint64_t *host_bytes,
                           uint64_t *arena_bytes_min, uint64_t *workspace_bytes) {
    if (!cfg) return KVS_ERR_INVALID;
    std::string why;
    if (!geometry_ok(cfg, &why)) {
        g_create_error = why;
        return KVS_ERR_UNSUPPORTED;
    }
    sizes_of(cfg, page_bytes, host_bytes, arena_bytes_min, workspace_bytes);
    return KVS_OK;
}

kvs_status kvs_create(const kvs_config *cfg, kvs_ctx **out) {
    if (!out) return KVS_ERR_INVALID;
    *out = nullptr;
    g_create_error.clear();
    if (!cfg) {
        g_create_error = "cfg is NULL";
        return KVS_ERR_INVALID;
    }
    std::string why;
    if (!geometry_ok(cfg, &why)) {
        g_create_error = why;
        return KVS_ERR_UNSUPPORTED;
    }
    uint64_t page_bytes, host_min, arena_min, ws_min;
    sizes_of(cfg, &page_bytes, &host_min, &arena_min, &ws_min);
    const bool plan_only = (cfg->flags & KVS_FLAG_PLAN_ONLY) != 0;
    if (cfg->ring_slots < 1) {
        g_create_error = "ring_slots must be >= 1";
        return KVS_ERR_INVALID;
    }
    if (cfg->n_lanes > 8) {
        g_create_error = "n_lanes must be 1..8";
        return KVS_ERR_INVALID;
    }
    if (!cfg->arena || cfg->arena_bytes < arena_min) {
        g_create_error = "arena below the minimum of 2 tail slots per layer plus the ring (" +
                         std::to_string(arena_min) + " bytes)";
        return KVS_ERR_ARENA;
    }
    if (!cfg->workspace || cfg->workspace_bytes < ws_min) {
        g_create_error = "workspace below the minimum (" + std::to_string(ws_min) + " bytes)";
        return KVS_ERR_ARENA;
    }
    if ((reinterpret_cast<uintptr_t>(cfg->arena) & 255) || (reinterpret_cast<uintptr_t>(cfg->workspace) & 255)) {
        g_create_error = "arena and workspace must be 256-byte aligned";
        return KVS_ERR_INVALID;
    }
    if ((!cfg->host && !plan_only) || cfg->host_bytes < host_min) {
        g_create_error = "host history below the minimum (" + std::to_string(host_min) + " bytes)";
        return KVS_ERR_HOST;
    }
    kvs_ctx *c = new kvs_ctx();
    c->cfg = *cfg;
    c->plan_only = plan_only;
    c->geom = kvs::make_geom((int)cfg->page_tokens, (int)cfg->n_kv_head, (int)cfg->head_dim);
    c->attn = static_cast<cudaStream_t>(cfg->attn_stream);
    c->copy = static_cast<cudaStream_t>(cfg->copy_stream);
    c->n_lanes = cfg->n_lanes ? (int)cfg->n_lanes : 1;
    c->lanes.assign(2 * c->n_lanes, nullptr);
    c->lanes[0] = c->attn;
    c->lanes[1] = c->copy;
    for (int l = 1; l < c->n_lanes; ++l) {
        c->lanes[2 * l] = static_cast<cudaStream_t>(cfg->lane_attn_streams[l - 1]);
        c->lanes[2 * l + 1] = static_cast<cudaStream_t>(cfg->lane_copy_streams[l - 1]);
    }
    c->max_pages = (int64_t)((cfg->max_tokens + cfg->page_tokens - 1) / cfg->page_tokens);
    c->page_pub_gen.assign((size_t)cfg->n_layers * (size_t)c->max_pages, 0);
    c->prefill_split = (int64_t)prefill_split_of(cfg);
    c->split_chunks = (uint64_t)cfg->max_q_head * cfg->max_rows > 64ull * cfg->n_kv_head &&
                      prefill_geometry(cfg->head_dim, cfg->page_tokens);
    c->verify_rows = (uint32_t)verify_rows_of(cfg);
    {
        const uint32_t G = cfg->max_q_head / cfg->n_kv_head;
        c->qfrag_groups = (int64_t)((c->verify_rows + rows_per_group(G) - 1) / rows_per_group(G));
    }
    c->layers.resize(cfg->n_layers);
    for (auto &L : c->layers) L.pool_slot.assign(c->max_pages, -1);
    c->n_slots = (int64_t)(cfg->arena_bytes / (uint64_t)c->geom.page_bytes);
    c->ring_n = cfg->ring_slots;
    c->chunk_pages = cfg->chunk_pages ? std::min(cfg->chunk_pages, cfg->ring_slots)
                                      : default_chunk_pages(cfg->ring_slots);
    c->ring_first = c->n_slots - c->ring_n;
    c->pool_n = c->ring_first - 2 * (int64_t)cfg->n_layers;
    c->pool_layer.assign(c->pool_n, -1);
    c->pool_page.assign(c->pool_n, -1);
    c->slot_last_chunk.assign(c->ring_n, -1);
    c->chunk_reader_sid.assign(c->ring_n, -1);
    memset(&c->st, 0, sizeof(c->st));
    c->host = static_cast<uint8_t *>(cfg->host);
    c->host_dev = c->host;
    if (!plan_only) {
        for (size_t i = 0; i < c->lanes.size(); ++i)
            for (size_t j = 0; j < i; ++j)
                if (!c->lanes[i] || c->lanes[i] == c->lanes[j]) {
                    delete c;
                    g_create_error = "attn/copy streams of all lanes must be distinct, non-null CUDA streams";
                    return KVS_ERR_INVALID;
                }
        cudaPointerAttributes pa;
        cudaError_t e = cudaPointerGetAttributes(&pa, cfg->host);
        if (e != cudaSuccess || pa.type != cudaMemoryTypeHost) {
            cudaGetLastError();
            e = cudaHostRegister(cfg->host, cfg->host_bytes, cudaHostRegisterMapped | cudaHostRegisterPortable);
            if (e != cudaSuccess) {
                cudaGetLastError();
                delete c;
                g_create_error = std::string("cudaHostRegister of the host history failed: ") + cudaGetErrorString(e);
                return KVS_ERR_HOST;
            }
            c->host_registered = true;
        }
        void *dp = nullptr;
        e = cudaHostGetDevicePointer(&dp, cfg->host, 0);
        if (e != cudaSuccess) {
            cudaGetLastError();
            if (c->host_registered) cudaHostUnregister(cfg->host);
            delete c;
            g_create_error = std::string("host history is not device-mapped: ") + cudaGetErrorString(e);
            return KVS_ERR_HOST;
        }
        c->host_dev = static_cast<uint8_t *>(dp);
    }
    c->lanes.push_back(nullptr);  // the resident-page stream
    c->lanes.push_back(nullptr);  // lane 0's ring-read stream
    if (!plan_only) {
        // resident pages of a layer that also reads ring chunks run beside
        // them at the lowest priority: ring reads gate the refills, resident
        // reads only fill the remaining SMs
        int least = 0, greatest = 0;
        cudaDeviceGetStreamPriorityRange(&least, &greatest);
        cudaError_t e = cudaStreamCreateWithPriority(&c->res_stream, cudaStreamNonBlocking, least);
        if (e != cudaSuccess) {
            c->res_stream = nullptr;
            if (c->host_registered) cudaHostUnregister(cfg->host);
            delete c;
            g_create_error = std::string("cudaStreamCreateWithPriority: ") + cudaGetErrorString(e);
            return KVS_ERR_CUDA;
        }
        c->lanes[c->res_sid()] = c->res_stream;
        e = cudaStreamCreateWithFlags(&c->ring0_stream, cudaStreamNonBlocking);
        if (e != cudaSuccess) {
            c->ring0_stream = nullptr;
            if (c->host_registered) cudaHostUnregister(cfg->host);
            delete c;
            g_create_error = std::string("cudaStreamCreateWithFlags: ") + cudaGetErrorString(e);
            return KVS_ERR_CUDA;
        }
        c->lanes[c->ring0_sid()] = c->ring0_stream;
    }
    if (create_events(c) != KVS_OK) {
        g_create_error = c->err;
        destroy_events(c);
        if (c->host_registered) cudaHostUnregister(cfg->host);
        delete c;
        return KVS_ERR_CUDA;
    }
    if (!plan_only) {
        cudaError_t e = cudaMemset(cfg->workspace, 0, kStatusBytes + kObsBytes);
        if (e != cudaSuccess) {
            g_create_error = std::string("workspace status clear: ") + cudaGetErrorString(e);
            destroy_events(c);
            if (c->host_registered) cudaHostUnregister(cfg->host);
            delete c;
            return KVS_ERR_CUDA;
        }
    }
    c->st.ring_slots = c->ring_n;
    c->st.chunk_pages = c->chunk_pages;
    c->st.pool_slots = (uint64_t)c->pool_n;
    *out = c;
    return KVS_OK;
}

kvs_status kvs_destroy(kvs_ctx *c) {
    if (!c) return KVS_ERR_INVALID;
    if (!c->plan_only) {
        for (cudaStream_t st : c->lanes) cudaStreamSynchronize(st);
        for (auto &t : c->timer_pending) {
            cudaEventDestroy(t.start);
            cudaEventDestroy(t.stop);
        }
        for (cudaEvent_t e : c->timer_free) cudaEventDestroy(e);
        release_graph(c);
        if (c->host_registered) cudaHostUnregister(c->cfg.host);
    }
    destroy_events(c);
    delete c;
    return KVS_OK;
}

kvs_status kvs_length(const kvs_ctx *c, uint32_t layer, uint64_t *n) {
    if (!c || !n || layer >= c->cfg.n_layers) return KVS_ERR_INVALID;
    *n = c->layers[layer].T;
    return KVS_OK;
}

kvs_status kvs_append(kvs_ctx *c, uint32_t layer, const float *k_dev, const float *v_dev,
                      uint32_t n_tokens) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    if (layer >= c->cfg.n_layers) return fail(c, KVS_ERR_INVALID, "layer out of range");
    if (n_tokens == 0) return KVS_OK;
    if (!c->plan_only && (!k_dev || !v_dev)) return fail(c, KVS_ERR_INVALID, "null K/V rows");
    LayerState &L = c->layers[layer];
    if (L.T + n_tokens > c->cfg.max_tokens) return fail(c, KVS_ERR_CAPACITY, "append beyond max_tokens");
    {
        kvs_status s0 = settle_clear(c, layer);
        if (s0 != KVS_OK) return s0;
    }
    const int P = c->geom.P;
    // Pre-check every eviction this append causes, so a refusal changes nothing.
    {
        int64_t free_pool = c->pool_n - c->pool_used;
        int64_t lease_free = c->lease_layer == (int64_t)layer ? (int64_t)c->lease_spare.size() : 0;
        for (uint64_t t = L.T; t < L.T + n_tokens; t = (t / P + 1) * P) {
            if (t % P != 0) continue;
            const int64_t q = (int64_t)(t / P), old = q - 2;
            if (old < 0 || L.tail_page[q & 1] != old) continue;
            if (evict_target(c, layer, old, free_pool) != 1 && lease_free > 0) {
                lease_free--;
                continue;
            }
            if (evict_target(c, layer, old, free_pool) < 0)
                return fail(c, KVS_ERR_STATE,
                            "append would move a page out of its tail slot while the layer has a pending "
                            "prefetch behind which other layers are queued, and the pool has no free slot");
            if (evict_target(c, layer, old, free_pool) == 1) free_pool--;
        }
    }
    uint64_t done = 0;
    while (done < n_tokens) {
        const uint64_t t = L.T;
        const int64_t q = (int64_t)(t / P);
        const int t0 = (int)(t % P);
        const uint32_t n = (uint32_t)std::min<uint64_t>(n_tokens - done, (uint64_t)(P - t0));
        const int64_t tslot = c->tail_slot(layer, q);
        kvs_status s;
        if (t0 != 0 && L.tail_page[q & 1] != q)
            return fail(c, KVS_ERR_STATE, "internal: the partial tail page is not in its tail slot");
        // a D2H publish of this slot may still be reading it
        s = op_wait(c, kAttn, c->ev_pub0 + (int)tslot);
        if (s != KVS_OK) return s;
        if (t0 == 0) {
            // page q starts in tail slot q % 2: evict its previous page
            const int64_t old = L.tail_page[q & 1];
            if (old >= 0 && old != q) {
                int target = evict_target(c, layer, old, c->pool_n - c->pool_used);
                // a page leaving a leased layer's tail extends the lease while it has spare slots
                if (target != 1 && c->lease_layer == (int64_t)layer && !c->lease_spare.empty()) target = 3;
                if (target == 3) {
                    const int64_t ls = c->lease_spare.back();
                    c->lease_spare.pop_back();
                    L.pool_slot[old] = ls;
                    if (c->plan_only) {
                        log_op(c, KVS_OP_MOVE, kAttn, layer, 0, old, ls);
                    } else {
                        cudaError_t e = cudaMemcpyAsync(c->slot_ptr(ls), c->slot_ptr(tslot), (size_t)c->geom.page_bytes,
                                                        cudaMemcpyDeviceToDevice, c->attn);
                        if (e != cudaSuccess) return cuda_fail(c, e, "tail -> lease move");
                    }
                } else if (target == 1) {
                    const int64_t ps = pool_alloc(c, layer, old);
                    L.pool_slot[old] = ps;
                    if (c->plan_only) {
                        log_op(c, KVS_OP_MOVE, kAttn, layer, 0, old, ps);
                    } else {
                        cudaError_t e = cudaMemcpyAsync(c->slot_ptr(ps), c->slot_ptr(tslot),
                                                        (size_t)c->geom.page_bytes,
                                                        cudaMemcpyDeviceToDevice, c->attn);
                        if (e != cudaSuccess) return cuda_fail(c, e, "tail -> pool move");
                    }
                } else if (target == 2) {
                    // stream it: it joins the pending plan of this (last announced) layer
                    Chunk ch;
                    ch.id = c->next_chunk++;
                    ch.layer = layer;
                    ch.seq0 = c->ring_seq++;
                    ch.pages.push_back(old);
                    c->queue.push_back(std::move(ch));
                }
            }
            L.tail_page[q & 1] = q;
            if (c->plan_only) {
                c->st.kernel_launches++;
            } else {
                cudaError_t e = kvs::launch_clear_tail(c->slot_ptr(tslot), c->geom, t0, c->attn,
                                                       tl_take(c, KVS_TL_CLEAR, layer, kAttn));
                if (e != cudaSuccess) return cuda_fail(c, e, "tail page clear");
                c->st.kernel_launches++;
            }
        }
        if (c->plan_only) {
            log_op(c, KVS_OP_WRITE, kAttn, layer, 0, q, tslot, n);
        } else {
            kvs::QuantizeParams qp;
            const int64_t row = (int64_t)c->geom.Hk * c->geom.D;
            qp.k = k_dev + (int64_t)done * row;
            qp.v = v_dev + (int64_t)done * row;
            qp.page = c->slot_ptr(tslot);
            qp.geom = c->geom;
            qp.t0 = t0;
            qp.n = (int)n;
            qp.tl = tl_take(c, KVS_TL_APPEND, layer, kAttn);
            cudaError_t e = kvs::launch_quantize(qp, c->attn);
            if (e != cudaSuccess) return cuda_fail(c, e, "quantise/append launch");
        }
        c->st.kernel_launches++;
        L.T += n;
        done += n;
        if (L.T % P == 0) {
            // page q is complete: publish it to the host history
            s = join_attn_into_copy(c);
            if (s != KVS_OK) return s;
            if (c->plan_only) {
                log_op(c, KVS_OP_PUBLISH, kCopy, layer, 0, q, tslot);
            } else {
                cudaError_t e = cudaMemcpyAsync(c->host_page(layer, q), c->slot_ptr(tslot),
                                                (size_t)c->geom.page_bytes, cudaMemcpyDeviceToHost,
                                                c->copy);
                if (e != cudaSuccess) return cuda_fail(c, e, "tail publish");
            }
            s = op_record(c, kCopy, c->ev_pub0 + (int)tslot);
            if (s != KVS_OK) return s;
            s = mark_publish(c, layer, q);
            if (s != KVS_OK) return s;
            c->st.d2h_pages++;
            c->st.d2h_bytes += (uint64_t)c->geom.page_bytes;
        }
    }
    return KVS_OK;
}

kvs_status kvs_truncate(kvs_ctx *c, uint32_t layer, uint64_t n_tokens) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    if (layer >= c->cfg.n_layers) return fail(c, KVS_ERR_INVALID, "layer out of range");
    LayerState &L = c->layers[layer];
    if (n_tokens > L.T) return fail(c, KVS_ERR_INVALID, "truncate beyond the current length");
    if (n_tokens == L.T) return KVS_OK;
    if (layer_has_plan(c, layer)) return fail(c, KVS_ERR_STATE, "layer has a pending prefetch");
    const int P = c->geom.P;
    const int64_t new_last = n_tokens ? (int64_t)((n_tokens - 1) / P) : -1;
    const int64_t cur_last = (int64_t)((L.T - 1) / P);
    // pages new_last+1 .. cur_last are dropped; the new tail page must be in a tail slot
    if (n_tokens > 0 && n_tokens % P != 0 && L.tail_page[new_last & 1] != new_last)
        return fail(c, KVS_ERR_UNSUPPORTED, "truncation further back than the two tail pages");
    for (int64_t p = new_last + 1; p <= cur_last; ++p) {
        if (L.tail_page[p & 1] == p) L.tail_page[p & 1] = -1;
        if (p < (int64_t)L.pool_slot.size() && L.pool_slot[p] >= 0) {
            if (is_lease_slot(c, L.pool_slot[p])) c->lease_spare.push_back(L.pool_slot[p]);
            pool_free(c, L.pool_slot[p]);
            L.pool_slot[p] = -1;
        }
    }
    if (n_tokens % P != 0 && !c->plan_only) {
        // on the resident-page stream, after everything enqueued on the
        // attention stream (this layer's reads) and after a publish of the slot
        const int rs = c->res_sid();
        const int64_t ts = c->tail_slot(layer, new_last);
        kvs_status s = join(c, kAttn, rs);
        if (s == KVS_OK) s = op_wait(c, rs, c->ev_pub0 + (int)ts);
        if (s != KVS_OK) return s;
        cudaError_t e = kvs::launch_clear_tail(c->slot_ptr(ts), c->geom, (int)(n_tokens % P), c->stream(rs),
                                               tl_take(c, KVS_TL_CLEAR, layer, rs));
        if (e != cudaSuccess) return cuda_fail(c, e, "truncate clear");
        c->st.kernel_launches++;
        s = op_record(c, rs, c->ev_clear0 + (int)layer);
        if (s != KVS_OK) return s;
        c->clear_pending[layer] = 1;
    }
    L.T = n_tokens;
    return KVS_OK;
}

// Pre-encoded complete pages straight into the host history (the authoritative
// copy of every page), extending a page-aligned layer.
kvs_status kvs_load_host_pages(kvs_ctx *c, uint32_t layer, uint64_t first_page, uint64_t n_pages,
                               const void *src) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    if (layer >= c->cfg.n_layers) return fail(c, KVS_ERR_INVALID, "layer out of range");
    if (c->capturing) return fail(c, KVS_ERR_STATE, "not allowed inside a step capture");
    if (!c->queue.empty() || !c->announced.empty())
        return fail(c, KVS_ERR_STATE, "host page load while prefetches are pending");
    if (c->lease_layer >= 0) return fail(c, KVS_ERR_STATE, "host page load while a lease is held");
    if (n_pages == 0) return KVS_OK;
    if (!src) return fail(c, KVS_ERR_INVALID, "null source pages");
    if (!c->host) return fail(c, KVS_ERR_STATE, "no host history");
    LayerState &L = c->layers[layer];
    const uint64_t P = (uint64_t)c->geom.P;
    if (L.T % P != 0 || first_page != L.T / P)
        return fail(c, KVS_ERR_INVALID, "loaded pages must continue a page-aligned history (first_page = T / P)");
    if (n_pages > (uint64_t)c->max_pages - first_page || (first_page + n_pages) * P > c->cfg.max_tokens)
        return fail(c, KVS_ERR_CAPACITY, "loaded pages reach beyond max_tokens");
    // a publish on the copy stream may still be writing the host history
    kvs_status s = kvs_sync(c, 0);
    if (s != KVS_OK) return s;
    if (c->graph_exec) {  // its captured lengths no longer hold
        release_graph(c);
        c->graph_kernels = 0;
    }
    // the tail slots give up their (complete, published) pages: to the pool
    // where the mask asks and there is room, else they are host-only
    for (int i = 0; i < 2; ++i) {
        const int64_t old = L.tail_page[i];
        if (old < 0) continue;
        if (evict_target(c, layer, old, c->pool_n - c->pool_used) == 1) {
            const int64_t ps = pool_alloc(c, layer, old);
            L.pool_slot[old] = ps;
            if (c->plan_only) {
                log_op(c, KVS_OP_MOVE, kAttn, layer, 0, old, ps);
            } else {
                cudaError_t e = cudaMemcpyAsync(c->slot_ptr(ps), c->slot_ptr(c->tail_slot(layer, old)),
                                                (size_t)c->geom.page_bytes, cudaMemcpyDeviceToDevice, c->attn);
                if (e != cudaSuccess) return cuda_fail(c, e, "tail -> pool move");
            }
        }
        L.tail_page[i] = -1;
    }
    const uint8_t *from = static_cast<const uint8_t *>(src);
    for (uint64_t i = 0; i < n_pages; ++i)
        memcpy(c->host_page(layer, (int64_t)(first_page + i)), from + i * (uint64_t)c->geom.page_bytes,
               (size_t)c->geom.page_bytes);
    L.T = (first_page + n_pages) * P;
    return KVS_OK;
}

kvs_status kvs_set_residency(kvs_ctx *c, uint32_t layer, const uint8_t *mask, uint64_t n_pages) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    if (c->capturing) return fail(c, KVS_ERR_STATE, "not allowed inside a step capture");
    if (layer >= c->cfg.n_layers) return fail(c, KVS_ERR_INVALID, "layer out of range");
    if (n_pages > (uint64_t)c->max_pages) return fail(c, KVS_ERR_INVALID, "mask longer than max pages");
    if (n_pages && !mask) return fail(c, KVS_ERR_INVALID, "null mask");
    if (!c->queue.empty() || !c->announced.empty())
        return fail(c, KVS_ERR_STATE, "residency change while prefetches are pending");
    if (c->lease_layer >= 0) return fail(c, KVS_ERR_STATE, "residency change while a lease is held");
    LayerState &L = c->layers[layer];
    const int64_t complete = (int64_t)(L.T / c->geom.P);  // pages 0..complete-1 are full
    {
        kvs_status s0 = settle_clear(c, layer);
        if (s0 != KVS_OK) return s0;
    }
    if (c->graph_exec) {  // its baked slot schedule no longer holds
        if (!c->plan_only) cudaStreamSynchronize(c->attn);
        release_graph(c);
        c->graph_kernels = 0;
    }
    std::vector<uint8_t> want(c->max_pages, 0);
    for (uint64_t i = 0; i < n_pages; ++i) want[i] = mask[i] ? 1 : 0;
    // count the change
    int64_t need = 0;
    for (int64_t p = 0; p < complete; ++p) {
        int64_t s;
        const int loc = locate(c, layer, p, &s);
        if (want[p] && loc == 0) need++;
        if (!want[p] && loc == 2) need--;
    }
    if (need > c->pool_n - c->pool_used)
        return fail(c, KVS_ERR_CAPACITY, "resident pool has too few free slots for this mask");
    L.mask.assign(want.begin(), want.begin() + std::max<int64_t>(n_pages, 0));
    // slots leaving the pool may still be read by queued attention
    kvs_status s = join_attn_lanes_into_attn(c);
    if (s != KVS_OK) return s;
    s = join_attn_into_copy(c);
    if (s != KVS_OK) return s;
    for (int64_t p = 0; p < complete; ++p) {
        if (!want[p] && L.pool_slot[p] >= 0 && L.tail_page[p & 1] != p) {
            pool_free(c, L.pool_slot[p]);
            L.pool_slot[p] = -1;
        }
    }
    std::vector<int64_t> pages, slots;
    for (int64_t p = 0; p < complete; ++p) {
        int64_t sl;
        if (want[p] && locate(c, layer, p, &sl) == 0) {
            const int64_t ps = pool_alloc(c, layer, p);
            L.pool_slot[p] = ps;
            pages.push_back(p);
            slots.push_back(ps);
        }
    }
    if (!pages.empty()) {
        s = op_copy_pages(c, layer, pages, slots, KVS_OP_POOL_LOAD, nullptr);
        if (s != KVS_OK) return s;
        c->st.pool_load_bytes += pages.size() * (uint64_t)c->geom.page_bytes;
        s = join_copy_into_attn(c);
        if (s != KVS_OK) return s;
    }
    return KVS_OK;
}

kvs_status kvs_set_ring_slots(kvs_ctx *c, uint32_t n_slots, uint32_t chunk_pages) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    if (c->capturing) return fail(c, KVS_ERR_STATE, "not allowed inside a step capture");
    if (n_slots < 1) return fail(c, KVS_ERR_INVALID, "ring needs at least one slot");
    if (!c->queue.empty() || !c->announced.empty())
        return fail(c, KVS_ERR_STATE, "ring change while prefetches are pending");
    if (c->lease_layer >= 0) return fail(c, KVS_ERR_STATE, "ring change while a lease is held");
    const int64_t base = 2 * (int64_t)c->cfg.n_layers;
    const int64_t new_pool = c->n_slots - base - (int64_t)n_slots;
    if (new_pool < 0) return fail(c, KVS_ERR_CAPACITY, "arena too small for that ring");
    if (c->pool_used > new_pool) return fail(c, KVS_ERR_CAPACITY, "resident pages exceed the new pool");
    // ring and pool slots change role: order after all earlier device work
    kvs_status s = join_all_into_attn(c);
    if (s != KVS_OK) return s;
    s = join_attn_into_copy(c);
    if (s != KVS_OK) return s;
    s = join_copy_into_attn(c);
    if (s != KVS_OK) return s;
    // compact resident pages that sit in slots the new ring takes
    for (int64_t i = new_pool; i < c->pool_n; ++i) {
        if (c->pool_layer[i] < 0) continue;
        int64_t j = 0;
        while (j < new_pool && c->pool_layer[j] >= 0) ++j;
        const uint32_t layer = (uint32_t)c->pool_layer[i];
        const int64_t page = c->pool_page[i];
        if (c->plan_only) {
            log_op(c, KVS_OP_MOVE, kAttn, layer, 0, page, c->pool_slot_id(j));
        } else {
            cudaError_t e = cudaMemcpyAsync(c->slot_ptr(c->pool_slot_id(j)), c->slot_ptr(c->pool_slot_id(i)),
                                            (size_t)c->geom.page_bytes, cudaMemcpyDeviceToDevice, c->attn);
            if (e != cudaSuccess) return cuda_fail(c, e, "pool compaction");
        }
        c->pool_layer[j] = c->pool_layer[i];
        c->pool_page[j] = page;
        c->pool_layer[i] = -1;
        c->pool_page[i] = -1;
        c->layers[layer].pool_slot[page] = c->pool_slot_id(j);
    }
    s = join_attn_into_copy(c);
    if (s != KVS_OK) return s;
    // new event set for the new ring size; a captured step graph is dropped
    if (!c->plan_only)
        for (cudaStream_t st : c->lanes) cudaStreamSynchronize(st);
    release_graph(c);
    c->graph_kernels = 0;
    destroy_events(c);
    c->ring_n = n_slots;
    c->chunk_pages = chunk_pages ? std::min(chunk_pages, n_slots) : default_chunk_pages(n_slots);
    c->ring_first = c->n_slots - n_slots;
    c->pool_layer.resize(new_pool);
    c->pool_page.resize(new_pool);
    if (new_pool > c->pool_n) {
        std::fill(c->pool_layer.begin() + c->pool_n, c->pool_layer.end(), -1);
        std::fill(c->pool_page.begin() + c->pool_n, c->pool_page.end(), -1);
    }
    c->pool_n = new_pool;
    c->slot_last_chunk.assign(c->ring_n, -1);
    c->chunk_reader_sid.assign(c->ring_n, -1);
    c->ring_seq = 0;
    c->st.ring_slots = c->ring_n;
    c->st.chunk_pages = c->chunk_pages;
    c->st.pool_slots = (uint64_t)c->pool_n;
    return create_events(c);
}

// Give the ring a new size at the same first slot (slots above it leave or
// rejoin the ring), after every earlier device use of the ring slots.
kvs_status resize_ring(kvs_ctx *c, uint32_t n_slots) {
    kvs_status s = join_all_into_attn(c);
    if (s != KVS_OK) return s;
    s = join_attn_into_copy(c);
    if (s != KVS_OK) return s;
    s = join_copy_into_attn(c);
    if (s != KVS_OK) return s;
    if (!c->plan_only)
        for (cudaStream_t st : c->lanes) cudaStreamSynchronize(st);
    release_graph(c);
    c->graph_kernels = 0;
    destroy_events(c);
    c->ring_n = n_slots;
    c->chunk_pages = std::min(c->chunk_pages, n_slots);
    c->slot_last_chunk.assign(c->ring_n, -1);
    c->chunk_reader_sid.assign(c->ring_n, -1);
    c->ring_seq = 0;
    c->st.ring_slots = c->ring_n;
    c->st.chunk_pages = c->chunk_pages;
    return create_events(c);
}

// Complete-layer lease: the layer's nonresident pages are loaded once into
// slots taken off the top of the ring (plus spare slots for pages that leave
// its tail while the lease is held); attention then reads them like resident
// pages, and the other layers stream through the smaller ring, so no refill
// can overwrite a leased slot until kvs_lease_release gives them back.
kvs_status kvs_lease_acquire(kvs_ctx *c, uint32_t layer, uint32_t extra_slots) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    if (layer >= c->cfg.n_layers) return fail(c, KVS_ERR_INVALID, "layer out of range");
    if (c->capturing) return fail(c, KVS_ERR_STATE, "not allowed inside a step capture");
    if (c->lease_layer >= 0) return fail(c, KVS_ERR_STATE, "a lease is already held");
    if (!c->queue.empty() || !c->announced.empty())
        return fail(c, KVS_ERR_STATE, "lease while prefetches are pending");
    {
        kvs_status s0 = settle_clear(c, layer);
        if (s0 != KVS_OK) return s0;
    }
    LayerState &L = c->layers[layer];
    std::vector<int64_t> pages;
    for (int64_t p = 0; p < n_pages_of(c, layer); ++p) {
        int64_t sl;
        if (locate(c, layer, p, &sl) == 0) pages.push_back(p);
    }
    const uint64_t k = pages.size() + (uint64_t)extra_slots;
    if (k >= c->ring_n)
        return fail(c, KVS_ERR_CAPACITY, "the lease needs " + std::to_string(k) + " ring slots and the ring (" +
                                             std::to_string(c->ring_n) + ") must keep at least one");
    const uint32_t full = c->ring_n;
    kvs_status s = resize_ring(c, full - (uint32_t)k);
    if (s != KVS_OK) return s;
    c->lease_layer = layer;
    c->lease_ring_full = full;
    std::vector<int64_t> slots;
    for (uint64_t i = 0; i < k; ++i) {
        const int64_t slot = c->ring_first + (int64_t)c->ring_n + (int64_t)i;
        if (i < pages.size()) {
            slots.push_back(slot);
            L.pool_slot[pages[i]] = slot;
        } else {
            c->lease_spare.push_back(slot);
        }
    }
    if (!pages.empty()) {
        s = op_copy_pages(c, layer, pages, slots, KVS_OP_POOL_LOAD, nullptr);
        if (s != KVS_OK) return s;
        c->st.pool_load_bytes += pages.size() * (uint64_t)c->geom.page_bytes;
        s = join_copy_into_attn(c);
        if (s != KVS_OK) return s;
    }
    return KVS_OK;
}

kvs_status kvs_lease_release(kvs_ctx *c) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    if (c->capturing) return fail(c, KVS_ERR_STATE, "not allowed inside a step capture");
    if (c->lease_layer < 0) return fail(c, KVS_ERR_STATE, "no lease is held");
    if (!c->queue.empty() || !c->announced.empty())
        return fail(c, KVS_ERR_STATE, "lease release while prefetches are pending");
    LayerState &L = c->layers[c->lease_layer];
    for (int64_t &sl : L.pool_slot)  // the host history keeps every leased page
        if (sl >= 0 && is_lease_slot(c, sl)) sl = -1;
    const uint32_t full = c->lease_ring_full;
    c->lease_layer = -1;
    c->lease_spare.clear();
    return resize_ring(c, full);
}

kvs_status kvs_lease_info(const kvs_ctx *c, int64_t *layer, uint32_t *leased_slots, uint32_t *spare_slots) {
    if (!c) return KVS_ERR_INVALID;
    if (layer) *layer = c->lease_layer;
    if (leased_slots) *leased_slots = c->lease_layer >= 0 ? c->lease_ring_full - c->ring_n : 0;
    if (spare_slots) *spare_slots = (uint32_t)c->lease_spare.size();
    return KVS_OK;
}

kvs_status kvs_prefetch(kvs_ctx *c, uint32_t layer) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    if (layer >= c->cfg.n_layers) return fail(c, KVS_ERR_INVALID, "layer out of range");
    if (layer_has_plan(c, layer)) return KVS_OK;
    plan_layer(c, layer);
    return pump(c);
}

// Prefill branch of kvs_attend: one tensor-core launch per batch of fully
// device-resident splits, then one per streamed split once all of its ring
// chunks are ready; each split's partial lands in its own row of the workspace.
kvs_status attend_prefill(kvs_ctx *c, uint32_t layer, const void *q_dev, uint32_t n_rows, uint32_t n_q_head,
                          uint64_t pos0, float scale, int64_t last, float *part_o, float *part_ml) {
    const int64_t SP = c->prefill_split;
    const int64_t n_split = last / SP + 1;
    kvs::PrefillParams pp;
    memset(&pp, 0, offsetof(kvs::PrefillParams, split_begin));
    pp.arena = static_cast<const uint8_t *>(c->cfg.arena);
    pp.geom = c->geom;
    pp.q = q_dev;
    pp.part_o = part_o;
    pp.part_ml = part_ml;
    pp.status = static_cast<int *>(c->cfg.workspace);
    pp.R = (int)n_rows;
    pp.Hq = (int)n_q_head;
    pp.G = (int)(n_q_head / c->geom.Hk);
    pp.pos0 = (long long)pos0;
    pp.scale_log2 = scale * 1.4426950408889634f;

    // (pages, slots) of one split; slot -1 where the page is in the ring
    auto split_pages = [&](int64_t sidx, std::vector<int64_t> &pg, std::vector<int64_t> &sl) {
        pg.clear();
        sl.clear();
        for (int64_t q = sidx * SP; q < std::min((sidx + 1) * SP, last + 1); ++q) {
            int64_t slot;
            const int kind = locate(c, layer, q, &slot);
            pg.push_back(q);
            sl.push_back(kind ? slot : -1);
        }
    };
    auto launch = [&](const std::vector<int64_t> &ids, const std::vector<std::vector<int64_t>> &pgs,
                      const std::vector<std::vector<int64_t>> &sls, uint32_t kind) -> kvs_status {
        c->st.kernel_launches++;
        c->st.decode_launches++;
        if (c->plan_only) {
            int64_t items = 0;
            for (auto &v : pgs) items += (int64_t)v.size();
            log_op(c, KVS_OP_LAUNCH, kAttn, layer, 0, 3, items);
            for (size_t i = 0; i < ids.size(); ++i)
                for (size_t j = 0; j < pgs[i].size(); ++j)
                    for (int g = 0; g < c->geom.Hk; ++g)
                        log_op(c, KVS_OP_READ, kAttn, layer, 0, pgs[i][j], sls[i][j], g);
            return KVS_OK;
        }
        pp.n_splits = (int)ids.size();
        int it = 0;
        for (size_t i = 0; i < ids.size(); ++i) {
            pp.split_begin[i] = it;
            pp.split_id[i] = (int)ids[i];
            for (size_t j = 0; j < pgs[i].size(); ++j, ++it) {
                pp.page[it] = (uint32_t)pgs[i][j];
                pp.slot[it] = (uint32_t)sls[i][j];
            }
        }
        pp.split_begin[ids.size()] = it;
        cudaEvent_t t0;
        kvs_status ts = timed_begin(c, kind, &t0, kAttn);
        if (ts != KVS_OK) return ts;
        pp.tl = tl_take(c, KVS_TL_PREFILL, layer, kAttn, (uint32_t)it);
        cudaError_t e = kvs::launch_prefill(pp, c->attn);
        if (e != cudaSuccess) return cuda_fail(c, e, "prefill kernel launch");
        c->check_status = true;
        return timed_end(c, t0, (uint64_t)it * (uint64_t)c->geom.page_bytes, kAttn);
    };

    kvs_status s = pump(c);
    if (s != KVS_OK) return s;
    // fully device-resident splits, batched
    {
        std::vector<int64_t> ids;
        std::vector<std::vector<int64_t>> pgs, sls;
        std::vector<int64_t> pg, sl;
        int items = 0;
        for (int64_t sidx = 0; sidx < n_split; ++sidx) {
            split_pages(sidx, pg, sl);
            if (std::find(sl.begin(), sl.end(), (int64_t)-1) != sl.end()) continue;
            if ((int)ids.size() == kvs::kMaxPrefillSplits || items + (int)pg.size() > kvs::kMaxPrefillItems) {
                s = launch(ids, pgs, sls, KVS_TIME_RESIDENT);
                if (s != KVS_OK) return s;
                ids.clear();
                pgs.clear();
                sls.clear();
                items = 0;
            }
            ids.push_back(sidx);
            pgs.push_back(pg);
            sls.push_back(sl);
            items += (int)pg.size();
            c->st.resident_pages_read += pg.size() * (uint64_t)c->geom.Hk;
        }
        if (!ids.empty()) {
            s = launch(ids, pgs, sls, KVS_TIME_RESIDENT);
            if (s != KVS_OK) return s;
        }
    }
    // streamed splits: all of a split's chunks ready, one launch, all released
    while (!c->queue.empty() && c->queue.front().layer == layer) {
        const int64_t sidx = c->queue.front().pages[0] / SP;
        std::vector<Chunk *> group;
        for (Chunk &ch : c->queue) {
            if (ch.layer != layer || ch.pages[0] / SP != sidx) break;
            group.push_back(&ch);
        }
        for (Chunk *ch : group) {
            if (!ch->filled) {
                s = pump(c);
                if (s != KVS_OK) return s;
                if (!ch->filled)
                    return fail(c, KVS_ERR_COVERAGE, "a prefill split's ring chunks do not fit in the ring together");
            }
            s = op_wait(c, kAttn, (int)(ch->id % c->ring_n));
            if (s != KVS_OK) return s;
        }
        if (sidx < n_split) {
            std::vector<int64_t> pg, sl;
            split_pages(sidx, pg, sl);
            for (Chunk *ch : group)
                for (size_t i = 0; i < ch->pages.size(); ++i)
                    for (size_t j = 0; j < pg.size(); ++j)
                        if (pg[j] == ch->pages[i]) sl[j] = c->ring_slot_id(ch->seq0 + i);
            s = launch({sidx}, {pg}, {sl}, KVS_TIME_RING);
            if (s != KVS_OK) return s;
            c->st.ring_pages_read += pg.size() * (uint64_t)c->geom.Hk;
        }
        for (Chunk *ch : group) {
            c->chunk_reader_sid[ch->id % c->ring_n] = kAttn;
            s = op_record(c, kAttn, (int)c->ring_n + (int)(ch->id % c->ring_n));
            if (s != KVS_OK) return s;
            c->attended = ch->id + 1;
            c->st.ring_chunks++;
        }
        for (size_t i = 0; i < group.size(); ++i) c->queue.pop_front();
        s = pump(c);
        if (s != KVS_OK) return s;
    }
    return KVS_OK;
}

kvs_status kvs_attend(kvs_ctx *c, uint32_t layer, const void *q_dev, int32_t q_dtype, uint32_t n_rows,
                      uint32_t n_q_head, uint64_t pos0, float scale, float *out_dev, float *lse_dev) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    if (layer >= c->cfg.n_layers) return fail(c, KVS_ERR_INVALID, "layer out of range");
    if (q_dtype != KVS_F32 && q_dtype != KVS_F16) return fail(c, KVS_ERR_INVALID, "q_dtype must be F32 or F16");
    if (n_rows < 1) return fail(c, KVS_ERR_INVALID, "n_rows must be >= 1");
    if (n_q_head < (uint32_t)c->geom.Hk || n_q_head % c->geom.Hk != 0 || n_q_head > c->cfg.max_q_head)
        return fail(c, KVS_ERR_INVALID, "n_q_head must be a multiple of n_kv_head and <= max_q_head");
    const uint32_t G = n_q_head / c->geom.Hk;
    if (n_rows > c->cfg.max_rows) return fail(c, KVS_ERR_UNSUPPORTED, "n_rows beyond max_rows");
    // more than 64 (row x head) per kv head: fp16 queries on a prefill-capable
    // geometry take the tensor-core path; any other call runs on the split-K
    // kernel as consecutive row groups, each group reading every staged span
    // before its ring slots are released
    const bool wide = G * n_rows > (uint32_t)kvs::decode_max_mma_rows();
    const bool prefill = wide && q_dtype == KVS_F16 && prefill_geometry(c->geom.D, c->geom.P);
    if (wide && !prefill && n_rows > c->verify_rows)
        return fail(c, KVS_ERR_UNSUPPORTED,
                    "a split-K call wider than 64 rows x heads per kv head needs n_rows <= max_verify_rows "
                    "(the workspace is sized for that many rows)");
    LayerState &L = c->layers[layer];
    if (pos0 + n_rows > L.T) return fail(c, KVS_ERR_CAPACITY, "rows beyond the appended length");
    if (!c->plan_only && (!q_dev || !out_dev)) return fail(c, KVS_ERR_INVALID, "null q or out");
    if (!c->announced.empty() && c->announced.front() != layer)
        return fail(c, KVS_ERR_STATE, "layers must be attended in the order they were prefetched");
    if (c->announced.empty()) plan_layer(c, layer);
    {
        kvs_status s0 = settle_clear(c, layer);
        if (s0 != KVS_OK) return s0;
    }

    const int P = c->geom.P;
    const int64_t last = (int64_t)((pos0 + n_rows - 1) / P);
    const int64_t np = n_pages_of(c, layer);

    // the plan must still cover exactly the nonresident pages
    std::vector<int64_t> res_pages, res_slots, streamed;
    for (int64_t p = 0; p < np; ++p) {
        int64_t s;
        if (locate(c, layer, p, &s) == 0) {
            streamed.push_back(p);
        } else if (p <= last) {
            res_pages.push_back(p);
            res_slots.push_back(s);
        }
    }
    {
        size_t k = 0;
        for (const Chunk &ch : c->queue) {
            if (ch.layer != layer) break;
            for (int64_t p : ch.pages) {
                if (k >= streamed.size() || streamed[k] != p)
                    return fail(c, KVS_ERR_COVERAGE, "span plan no longer matches the layer's residency");
                ++k;
            }
        }
        if (k != streamed.size()) return fail(c, KVS_ERR_COVERAGE, "span plan leaves nonresident pages uncovered");
    }

    const size_t per_split = (size_t)n_q_head * n_rows;
    uint8_t *qfrag = static_cast<uint8_t *>(c->cfg.workspace) + kStatusBytes + kObsBytes;
    const int64_t qf_bytes = kvs::qfrag_bytes(c->geom.Hk, c->geom.D);
    float *part_o = reinterpret_cast<float *>(qfrag + c->qfrag_groups * qf_bytes);
    const int64_t n_partials = prefill ? (c->max_pages + c->prefill_split - 1) / c->prefill_split : c->max_pages;
    float *part_ml = part_o + (size_t)n_partials * per_split * c->geom.D;
    c->st.attend_calls++;
    kvs_status s;
    if (prefill) {
        s = attend_prefill(c, layer, q_dev, n_rows, n_q_head, pos0, scale, last, part_o, part_ml);
        if (s != KVS_OK) return s;
    } else {
        kvs::DecodeParams dp;
        memset(&dp, 0, offsetof(kvs::DecodeParams, page));
        dp.arena = static_cast<const uint8_t *>(c->cfg.arena);
        dp.geom = c->geom;
        dp.q = q_dev;
        dp.q_f16 = q_dtype == KVS_F16;
        dp.part_o = part_o;
        dp.part_ml = part_ml;
        dp.status = static_cast<int *>(c->cfg.workspace);
        dp.qf = reinterpret_cast<const uint4 *>(qfrag);
        dp.R = (int)n_rows;
        dp.Hq = (int)n_q_head;
        dp.G = (int)G;
        dp.pos0 = (long long)pos0;
        dp.scale_log2 = scale * 1.4426950408889634f;
        dp.single_f16 = (c->cfg.flags & KVS_FLAG_F16_OPERANDS) ? 1 : 0;
        if (c->fault == KVS_FAULT_DEVICE_WAIT && c->fault_nth && ++c->fault_count == c->fault_nth)
            dp.give_up_waits = 1;
        // row groups: query rows row0 .. row0 + Rg - 1, G * Rg <= 64, each with its
        // own query fragments
        const uint32_t rpg = rows_per_group(G);
        std::vector<kvs::DecodeParams> groups;
        for (uint32_t r0 = 0; r0 < n_rows; r0 += rpg) {
            kvs::DecodeParams gp = dp;
            gp.row0 = (int)r0;
            gp.Rg = (int)std::min(rpg, n_rows - r0);
            gp.qf = reinterpret_cast<const uint4 *>(qfrag + (int64_t)groups.size() * qf_bytes);
            groups.push_back(gp);
        }

        // Q fragments for every kv head and row group, once per call (primary attention stream)
        for (kvs::DecodeParams &gp : groups) {
            c->st.kernel_launches++;
            if (c->plan_only) {
                log_op(c, KVS_OP_LAUNCH, kAttn, layer, 0, 4, c->geom.Hk);
            } else {
                gp.prep_q = 1;
                gp.n_items = 0;
                gp.tl_prep = tl_take(c, KVS_TL_QPREP, layer, kAttn);
                cudaError_t e = kvs::launch_decode(gp, c->attn);
                gp.tl_prep = nullptr;
                if (e != cudaSuccess) return cuda_fail(c, e, "query fragment launch");
                gp.prep_q = 0;
            }
        }
        // other lanes start after this call's inputs (Q and its fragments, the
        // previous combine's reads of the partials, published pages) are in place
        s = fork_attn_lanes(c);
        if (s != KVS_OK) return s;
        s = pump(c);
        if (s != KVS_OK) return s;
        // resident and tail pages need no fence.  When the layer also reads
        // ring chunks they go to the low-priority resident stream and leave
        // room (two chunk-read CTAs per SM) for the chunk reads in flight:
        // lanes x chunk pages x kv heads x row tiles.
        if (!res_pages.empty()) {
            const bool ring_too = !c->queue.empty() && c->queue.front().layer == layer;
            int sid = kAttn;
            int max_sms = 0;
            if (ring_too) {
                sid = c->res_sid();
                const int n_sms = kvs::current_device_sms();
                const int64_t ring_ctas =
                    (int64_t)c->n_lanes * c->chunk_pages * c->geom.Hk * ((G * std::min(rpg, n_rows) + 7) / 8);
                max_sms = n_sms - (int)std::min<int64_t>((ring_ctas + 1) / 2, n_sms / 3);
            }
            for (kvs::DecodeParams &gp : groups) {
                gp.max_sms = max_sms;
                s = launch_items(c, layer, res_pages, res_slots, gp, KVS_TIME_RESIDENT, sid);
                gp.max_sms = 0;
                if (s != KVS_OK) return s;
            }
            c->st.resident_pages_read += res_pages.size() * (uint64_t)c->geom.Hk;
        }
        // ring chunks in order: ready fence, read, consumed fence, refill
        std::vector<int64_t> last_read(c->n_lanes, -1);  // per lane: last chunk read in this call
        int chunk_in_layer = 0;
        while (!c->queue.empty() && c->queue.front().layer == layer) {
            Chunk &ch = c->queue.front();
            if (!ch.filled) {
                s = pump(c);
                if (s != KVS_OK) return s;
                if (!ch.filled) return fail(c, KVS_ERR_COVERAGE, "ring chunk could not be scheduled");
            }
            const int lane = (int)(ch.id % (uint64_t)c->n_lanes);
            const int sid = c->attn_sid_of_lane(lane);  // this chunk's attention stream
            s = op_wait(c, sid, (int)(ch.id % c->ring_n));
            if (s != KVS_OK) return s;
            // Stagger the lanes: the layer's first chunks are all in the ring when
            // it starts; read at once, their refills would run side by side and
            // the lanes would stay in phase (every lane reading while the link
            // idles, then every lane refilling at a share of the link).  Each of
            // the first n_lanes - 1 later chunks waits for the read before it, so a
            // lane reads while the previous lane's refill has the link.
            if (chunk_in_layer > 0 && chunk_in_layer < c->n_lanes) {
                s = op_wait(c, sid, (int)c->ring_n + (int)((ch.id - 1) % c->ring_n));
                if (s != KVS_OK) return s;
            }
            ++chunk_in_layer;
            std::vector<int64_t> pg, sl;
            for (size_t i = 0; i < ch.pages.size(); ++i) {
                if (ch.pages[i] > last) continue;
                pg.push_back(ch.pages[i]);
                sl.push_back(c->ring_slot_id(ch.seq0 + i));
            }
            if (!pg.empty()) {
                // every row group reads the chunk before its consumed fence; the
                // first accounts the chunk's wait for its copy
                for (size_t gi = 0; gi < groups.size(); ++gi) {
                    kvs::DecodeParams &gp = groups[gi];
                    if (gi == 0) {
                        gp.rec = obs_record(c, ch.id);
                        gp.acc = obs_accumulator(c);
                        gp.rec_pages = (int)pg.size();
                    }
                    s = launch_items(c, layer, pg, sl, gp, KVS_TIME_RING, sid);
                    gp.rec = nullptr;
                    gp.acc = nullptr;
                    if (s != KVS_OK) return s;
                }
                c->st.ring_pages_read += pg.size() * (uint64_t)c->geom.Hk;
            }
            c->chunk_reader_sid[ch.id % c->ring_n] = sid;
            s = op_record(c, sid, (int)c->ring_n + (int)(ch.id % c->ring_n));
            if (s != KVS_OK) return s;
            last_read[lane] = (int64_t)ch.id;
            c->attended = ch.id + 1;
            c->st.ring_chunks++;
            c->queue.pop_front();
            s = pump(c);
            if (s != KVS_OK) return s;
        }
        // The combine waits for this layer's reads only: each lane's last
        // consumed event (recorded before any refill went onto that lane) and
        // the resident-page stream; not for refills queued behind the reads.
        for (int l = 0; l < c->n_lanes; ++l) {
            if (last_read[l] < 0) continue;
            s = op_wait(c, kAttn, (int)c->ring_n + (int)(last_read[l] % c->ring_n));
            if (s != KVS_OK) return s;
        }
        s = join(c, c->res_sid(), kAttn);
        if (s != KVS_OK) return s;
    }
    c->announced.pop_front();
    // final reduction over splits in logical order
    c->st.kernel_launches++;
    if (c->plan_only) {
        log_op(c, KVS_OP_LAUNCH, kAttn, layer, 0, 2, (int64_t)n_rows * n_q_head);
    } else {
        kvs::CombineParams cp;
        cp.part_o = part_o;
        cp.part_ml = part_ml;
        cp.status = static_cast<const int *>(c->cfg.workspace);
        cp.out = out_dev;
        cp.lse = lse_dev;
        cp.R = (int)n_rows;
        cp.Hq = (int)n_q_head;
        cp.D = c->geom.D;
        cp.P = P;
        cp.split_pages = prefill ? (int)c->prefill_split : 1;
        cp.pos0 = (long long)pos0;
        cp.tl = tl_take(c, KVS_TL_COMBINE, layer, kAttn);
        cudaError_t e = kvs::launch_combine(cp, c->attn);
        if (e != cudaSuccess) return cuda_fail(c, e, "combine launch");
    }
    return pump(c);
}

kvs_status kvs_sync(kvs_ctx *c, uint32_t timeout_ms) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    if (c->capturing) return fail(c, KVS_ERR_STATE, "kvs_sync inside a step capture");
    const auto t0 = std::chrono::steady_clock::now();
    auto expired = [&]() {
        return timeout_ms && std::chrono::steady_clock::now() - t0 >= std::chrono::milliseconds(timeout_ms);
    };
    const bool stall = c->fault == KVS_FAULT_SYNC_STALL && c->fault_nth && ++c->fault_count >= c->fault_nth;
    if (c->plan_only) {
        if (!stall) return KVS_OK;
        while (!expired()) std::this_thread::sleep_for(std::chrono::microseconds(200));
        return fail(c, KVS_ERR_TIMEOUT, "kvs_sync deadline passed");
    }
    for (int sid = 0; sid < c->n_streams(); ++sid) {
        kvs_status s = op_record(c, sid, c->ev_lane0 + sid);
        if (s != KVS_OK) return s;
    }
    for (;;) {
        bool done = !stall;
        for (int sid = 0; sid < c->n_streams(); ++sid) {
            const int ev = c->ev_lane0 + sid;
            cudaError_t e = cudaEventQuery(c->events[ev]);
            if (e == cudaErrorNotReady) {
                done = false;
            } else if (e != cudaSuccess) {
                return cuda_fail(c, e, "kvs_sync");
            }
        }
        if (done) break;
        if (expired()) return fail(c, KVS_ERR_TIMEOUT, "kvs_sync deadline passed");
        std::this_thread::sleep_for(std::chrono::microseconds(20));
    }
    harvest_timers(c);
    std::fill(c->clear_pending.begin(), c->clear_pending.end(), 0);  // every stream has drained
    if (c->check_status) {
        c->check_status = false;
        int status = 0;
        cudaError_t e = cudaMemcpy(&status, c->cfg.workspace, sizeof(int), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(c, e, "status read");
        if (status != 0) {
            cudaMemset(c->cfg.workspace, 0, sizeof(int));
            return fail(c, KVS_ERR_CUDA, "a bounded device-side wait in an attention kernel timed out");
        }
    }
    return KVS_OK;
}

kvs_status kvs_flush(kvs_ctx *c, uint32_t layer) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    uint32_t l0 = layer, l1 = layer + 1;
    if (layer == UINT32_MAX) {
        l0 = 0;
        l1 = c->cfg.n_layers;
    } else if (layer >= c->cfg.n_layers) {
        return fail(c, KVS_ERR_INVALID, "layer out of range");
    }
    kvs_status s = settle_clears(c, l0, l1);
    if (s == KVS_OK) s = join_attn_into_copy(c);
    if (s != KVS_OK) return s;
    for (uint32_t l = l0; l < l1; ++l) {
        const LayerState &L = c->layers[l];
        if (L.T % c->geom.P == 0) continue;  // full pages were published already
        const int64_t q = (int64_t)(L.T / c->geom.P);
        const int64_t ts = c->tail_slot(l, q);
        if (c->plan_only) {
            log_op(c, KVS_OP_PUBLISH, kCopy, l, 0, q, ts);
        } else {
            cudaError_t e = cudaMemcpyAsync(c->host_page(l, q), c->slot_ptr(ts), (size_t)c->geom.page_bytes,
                                            cudaMemcpyDeviceToHost, c->copy);
            if (e != cudaSuccess) return cuda_fail(c, e, "tail flush");
        }
        s = op_record(c, kCopy, c->ev_pub0 + (int)ts);
        if (s != KVS_OK) return s;
        s = mark_publish(c, l, q);
        if (s != KVS_OK) return s;
        c->st.d2h_pages++;
        c->st.d2h_bytes += (uint64_t)c->geom.page_bytes;
    }
    return KVS_OK;
}

kvs_status kvs_page_location(const kvs_ctx *c, uint32_t layer, uint64_t page, int32_t *kind, int64_t *slot) {
    if (!c || !kind || !slot || layer >= c->cfg.n_layers || page >= (uint64_t)c->max_pages) return KVS_ERR_INVALID;
    *kind = locate(c, layer, (int64_t)page, slot);
    if (*kind == 2 && is_lease_slot(c, *slot)) *kind = 3;
    return KVS_OK;
}

kvs_status kvs_read_slot(kvs_ctx *c, int64_t slot, void *host_dst) {
    if (!c || !host_dst) return KVS_ERR_INVALID;
    if (c->capturing) return fail(c, KVS_ERR_STATE, "not allowed inside a step capture");
    if (slot < 0 || slot >= c->n_slots) return fail(c, KVS_ERR_INVALID, "slot out of range");
    if (c->plan_only) return fail(c, KVS_ERR_STATE, "no device memory in plan-only mode");
    kvs_status s = kvs_sync(c, 0);
    if (s != KVS_OK) return s;
    cudaError_t e = cudaMemcpy(host_dst, c->slot_ptr(slot), (size_t)c->geom.page_bytes, cudaMemcpyDeviceToHost);
    return e == cudaSuccess ? KVS_OK : cuda_fail(c, e, "slot read");
}

kvs_status kvs_read_host_page(kvs_ctx *c, uint32_t layer, uint64_t page, void *host_dst) {
    if (!c || !host_dst || layer >= c->cfg.n_layers || page >= (uint64_t)c->max_pages) return KVS_ERR_INVALID;
    if (c->capturing) return fail(c, KVS_ERR_STATE, "not allowed inside a step capture");
    if (!c->host) return fail(c, KVS_ERR_STATE, "no host history");
    kvs_status s = kvs_sync(c, 0);
    if (s != KVS_OK) return s;
    memcpy(host_dst, c->host_page(layer, (int64_t)page), (size_t)c->geom.page_bytes);
    return KVS_OK;
}

kvs_status kvs_ring_info(const kvs_ctx *c, int64_t *first_slot, uint32_t *n_slots) {
    if (!c) return KVS_ERR_INVALID;
    if (first_slot) *first_slot = c->ring_first;
    if (n_slots) *n_slots = c->ring_n;
    return KVS_OK;
}

kvs_status kvs_stats(kvs_ctx *c, kvs_stats_t *out, int reset) {
    if (!c || !out) return KVS_ERR_INVALID;
    if (!c->plan_only) harvest_timers(c);
    c->st.ring_slots = c->ring_n;
    c->st.chunk_pages = c->chunk_pages;
    c->st.pool_slots = (uint64_t)c->pool_n;
    c->st.pool_used = (uint64_t)c->pool_used;
    c->st.observed_reads = c->last_obs.streamed_reads;
    c->st.ready_misses = c->last_obs.ready_misses;
    c->st.ring_occupancy = c->last_obs.ring_occupancy;
    c->st.copy_busy = c->last_obs.copy_busy;
    *out = c->st;
    if (reset) {
        const uint64_t rs = c->st.ring_slots, ps = c->st.pool_slots, pu = c->st.pool_used;
        memset(&c->st, 0, sizeof(c->st));
        c->st.ring_slots = rs;
        c->st.pool_slots = ps;
        c->st.pool_used = pu;
    }
    return KVS_OK;
}

kvs_status kvs_observe(kvs_ctx *c, kvs_policy_observation *out, int reset) {
    if (!c || !out) return KVS_ERR_INVALID;
    c->err.clear();
    if (c->capturing) return fail(c, KVS_ERR_STATE, "not allowed inside a step capture");
    memset(out, 0, sizeof(*out));
    for (const LayerState &L : c->layers) out->context_tokens = std::max<uint64_t>(out->context_tokens, L.T);
    if (c->plan_only) return KVS_OK;
    kvs_status s = kvs_sync(c, 0);
    if (s != KVS_OK) return s;
    kvs::ObsAccumulator a;
    cudaError_t e = cudaMemcpy(&a, obs_accumulator(c), sizeof(a), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(c, e, "observation read");
    out->streamed_reads = a.reads;
    out->ready_misses = a.misses;
    const unsigned long long first = ~a.first_fill_neg;
    if (a.reads && a.last_read > first) {
        const double span = (double)(a.last_read - first);
        out->ring_occupancy = (float)std::min(1.0, (double)a.occupancy_page_ns / (span * (double)c->ring_n));
        out->copy_busy = (float)std::min(1.0, (double)a.fill_busy_ns / span);
        out->copy_bytes = a.fill_bytes;
        out->interval_ns = a.last_read - first;
    }
    c->last_obs = *out;
    if (reset) {
        e = cudaMemset(obs_accumulator(c), 0, sizeof(a));
        if (e != cudaSuccess) return cuda_fail(c, e, "observation reset");
    }
    return KVS_OK;
}

kvs_status kvs_timeline_begin(kvs_ctx *c, void *records_dev, uint32_t max_records) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    if (!c->plan_only && max_records > 0 && (!records_dev || (reinterpret_cast<uintptr_t>(records_dev) & 7u)))
        return fail(c, KVS_ERR_INVALID, "timeline records must be a non-null, 8-byte aligned device buffer");
    c->tl_buf = static_cast<unsigned long long *>(records_dev);
    c->tl_max = max_records;
    c->tl_dropped = 0;
    c->tl_meta.clear();
    c->tl_on = true;
    return KVS_OK;
}

kvs_status kvs_timeline_end(kvs_ctx *c) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    c->tl_on = false;
    return KVS_OK;
}

kvs_status kvs_timeline_read(kvs_ctx *c, kvs_timeline_record *out, uint32_t max_out, uint32_t *n_out,
                             uint32_t *n_dropped) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    const uint32_t n = (uint32_t)std::min<size_t>(max_out, c->tl_meta.size());
    if (n_out) *n_out = n;
    if (n_dropped) *n_dropped = c->tl_dropped;
    if (n == 0) return KVS_OK;
    if (!out) return fail(c, KVS_ERR_INVALID, "null output records");
    std::vector<unsigned long long> raw(2 * (size_t)n, 0ull);
    if (!c->plan_only) {
        cudaError_t e = cudaMemcpy(raw.data(), c->tl_buf, raw.size() * sizeof(unsigned long long),
                                   cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(c, e, "timeline read");
    }
    for (uint32_t i = 0; i < n; ++i) {
        out[i] = c->tl_meta[i];
        out[i].start_ns = raw[2 * i] ? ~raw[2 * i] : 0ull;
        out[i].end_ns = raw[2 * i + 1];
    }
    return KVS_OK;
}

kvs_status kvs_set_timing(kvs_ctx *c, int mask) {
    if (!c) return KVS_ERR_INVALID;
    c->timing = (uint32_t)mask & (KVS_TIME_RESIDENT | KVS_TIME_RING);
    return KVS_OK;
}

kvs_status kvs_graph_begin(kvs_ctx *c) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    if (c->capturing) return fail(c, KVS_ERR_STATE, "a step capture is already open");
    if (!c->queue.empty() || !c->announced.empty())
        return fail(c, KVS_ERR_STATE, "step capture must start with no prefetch pending");
    if (!c->plan_only) {
        // the graph records its own events: an event recorded inside a capture
        // cannot be waited on by work outside it
        std::vector<cudaEvent_t> fresh(c->events.size(), nullptr);
        for (auto &e : fresh) {
            cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
            if (r != cudaSuccess) {
                for (cudaEvent_t x : fresh)
                    if (x) cudaEventDestroy(x);
                return cuda_fail(c, r, "cudaEventCreate");
            }
        }
        cudaError_t e = cudaStreamBeginCapture(c->attn, cudaStreamCaptureModeRelaxed);
        if (e != cudaSuccess) {
            for (cudaEvent_t x : fresh) cudaEventDestroy(x);
            return cuda_fail(c, e, "cudaStreamBeginCapture");
        }
        c->eager_events.swap(c->events);
        c->events.swap(fresh);
    }
    c->capturing = true;
    c->ev_in_capture.assign(c->events.size(), 0);
    // inside the graph the ring starts empty: its earlier readers are ordered
    // before every replay by the join in kvs_graph_launch
    std::fill(c->slot_last_chunk.begin(), c->slot_last_chunk.end(), -1);
    c->graph_kernel_base = c->st.kernel_launches;
    kvs_status s = join_attn_into_copy(c);  // the copy stream joins the capture
    return s != KVS_OK ? s : fork_lanes(c);  // and so do the other lanes
}

kvs_status kvs_graph_end(kvs_ctx *c) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    if (!c->capturing) return fail(c, KVS_ERR_STATE, "no step capture is open");
    const bool pending = !c->queue.empty() || !c->announced.empty();
    kvs_status s = join_all_into_attn(c);  // every lane rejoins before capture ends
    c->capturing = false;
    cudaGraph_t g = nullptr;
    std::vector<cudaEvent_t> cap_events;
    if (!c->plan_only) {
        cudaError_t e = cudaStreamEndCapture(c->attn, &g);
        if (s == KVS_OK && e != cudaSuccess) s = cuda_fail(c, e, "cudaStreamEndCapture");
        cap_events.swap(c->events);
        c->events.swap(c->eager_events);
    }
    if (s == KVS_OK && pending) s = fail(c, KVS_ERR_STATE, "step capture ended with a prefetch pending");
    auto drop = [&]() {
        if (g) cudaGraphDestroy(g);
        for (cudaEvent_t x : cap_events)
            if (x) cudaEventDestroy(x);
    };
    if (s != KVS_OK) {
        drop();
        return s;
    }
    if (!c->plan_only) {
        cudaGraphExec_t ex = nullptr;
        cudaError_t e = cudaGraphInstantiate(&ex, g, 0);
        if (e != cudaSuccess) {
            drop();
            return cuda_fail(c, e, "cudaGraphInstantiate");
        }
        release_graph(c);
        c->graph = g;
        c->graph_exec = ex;
        c->graph_events.swap(cap_events);
    }
    c->graph_kernels = c->st.kernel_launches - c->graph_kernel_base;
    c->st.graph_kernels = c->graph_kernels;
    std::fill(c->slot_last_chunk.begin(), c->slot_last_chunk.end(), -1);
    return KVS_OK;
}

kvs_status kvs_graph_launch(kvs_ctx *c) {
    if (!c) return KVS_ERR_INVALID;
    c->err.clear();
    if (c->capturing) return fail(c, KVS_ERR_STATE, "cannot replay while capturing");
    if (!c->graph_exec && !c->plan_only) return fail(c, KVS_ERR_STATE, "no step graph captured");
    if (!c->queue.empty() || !c->announced.empty())
        return fail(c, KVS_ERR_STATE, "replay with a prefetch pending");
    kvs_status s = join_all_into_attn(c);
    if (s != KVS_OK) return s;
    if (!c->plan_only) {
        cudaError_t e = cudaGraphLaunch(c->graph_exec, c->attn);
        if (e != cudaSuccess) return cuda_fail(c, e, "cudaGraphLaunch");
    }
    c->st.graph_launches++;
    c->st.kernel_launches += c->graph_kernels;
    // later work on every lane waits for the replay's ring readers
    s = join_attn_into_copy(c);
    return s != KVS_OK ? s : fork_lanes(c);
}

kvs_status kvs_graph_destroy(kvs_ctx *c) {
    if (!c) return KVS_ERR_INVALID;
    if (c->capturing) return fail(c, KVS_ERR_STATE, "a step capture is open");
    if (!c->plan_only) cudaStreamSynchronize(c->attn);
    release_graph(c);
    c->graph_kernels = 0;
    return KVS_OK;
}


kvs_status kvs_debug_inject(kvs_ctx *c, uint32_t fault, uint64_t nth) {
    if (!c) return KVS_ERR_INVALID;
    if (fault > KVS_FAULT_DEVICE_WAIT) return fail(c, KVS_ERR_INVALID, "unknown fault kind");
    c->fault = nth ? fault : (uint32_t)KVS_FAULT_NONE;
    c->fault_nth = nth;
    c->fault_count = 0;
    return KVS_OK;
}

kvs_status kvs_trace_read(const kvs_ctx *c, uint64_t first, uint64_t max, kvs_trace_op *ops,
                          uint64_t *n_out, uint64_t *n_total) {
    if (!c) return KVS_ERR_INVALID;
    if (!c->plan_only) return KVS_ERR_STATE;
    const uint64_t n = c->trace.size();
    if (n_total) *n_total = n;
    uint64_t k = 0;
    if (ops)
        for (uint64_t i = first; i < n && k < max; ++i, ++k) ops[k] = c->trace[i];
    if (n_out) *n_out = k;
    return KVS_OK;
}

}  // extern "C"
