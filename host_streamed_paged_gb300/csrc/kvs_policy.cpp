// Adaptive residency policy: proposes how a fixed budget of page slots is
// split between resident pages and the shared ring.
//
// Design source: Adaptive KV Streaming for llama.cpp V2, "KV data movement
// and attention" (the split reacts to reads that waited on copies, to how
// full the ring runs and to how busy the copy stream is, and only after
// consistent evidence) and "Logical KV layout, policy, and physical
// execution" (a proposal computed from the context length and that
// feedback; applying it is a separate step that moves the bytes);
// Adaptive KV Streaming for llama.cpp, "Adaptive KV streaming" (as the
// context grows, resident space is kept as large as the budget allows and is
// handed to a larger ring gradually).  The pages name the inputs but no
// thresholds or step sizes; those come from kvs_policy_config.
//
// Pure host code: no context, no CUDA call, no allocation.
#include <stdint.h>

#include "kvs.h"

namespace {

bool fraction(float x) { return x >= 0.f && x <= 1.f; }  // false for NaN too

uint32_t clamp_u32(uint64_t x, uint32_t lo, uint32_t hi) {
    return x < lo ? lo : (x > hi ? hi : (uint32_t)x);
}

}  // namespace

extern "C" kvs_status kvs_policy_step(const kvs_policy_config *cfg, const kvs_policy_state *prev,
                                      const kvs_policy_observation *obs, kvs_policy_state *next,
                                      kvs_policy_decision *out) {
    if (!cfg || !prev || !obs || !next || !out) return KVS_ERR_INVALID;
    if (cfg->page_tokens == 0 || cfg->n_layers == 0 || cfg->budget_slots == 0 || cfg->step_slots == 0 ||
        cfg->hold_steps == 0)
        return KVS_ERR_INVALID;
    const uint32_t hi_cfg = cfg->max_ring_slots ? cfg->max_ring_slots : cfg->budget_slots;
    const uint32_t hi = hi_cfg < cfg->budget_slots ? hi_cfg : cfg->budget_slots;
    const uint32_t lo = cfg->min_ring_slots;
    if (lo == 0 || lo > hi) return KVS_ERR_INVALID;
    if (!fraction(cfg->miss_grow) || !fraction(cfg->copy_busy_max) || !fraction(cfg->occupancy_shrink) ||
        !fraction(obs->ring_occupancy) || !fraction(obs->copy_busy) || obs->ready_misses > obs->streamed_reads ||
        !(cfg->link_gbs >= 0.f && cfg->link_gbs < 1e9f))
        return KVS_ERR_INVALID;

    const uint64_t ppl = obs->context_tokens / cfg->page_tokens + (obs->context_tokens % cfg->page_tokens != 0);
    // the whole history (ppl pages in each layer) fits next to the smallest
    // ring: ppl * n_layers <= budget - lo, written without the product
    const bool fits = ppl <= (uint64_t)(cfg->budget_slots - lo) / cfg->n_layers;

    kvs_policy_state st = *prev;
    st.steps = prev->steps + 1;
    uint32_t ring;
    uint32_t reason;
    if (fits) {
        ring = lo;
        reason = KVS_POLICY_FITS;
        st.grow_run = st.shrink_run = 0;
    } else if (prev->ring_slots == 0) {
        ring = lo;
        reason = KVS_POLICY_INIT;
        st.grow_run = st.shrink_run = 0;
    } else {
        const double miss_rate = obs->streamed_reads ? (double)obs->ready_misses / (double)obs->streamed_reads : 0.0;
        // the link has room: its measured rate against the caller's ceiling when both
        // are known (refills of several lanes overlap, so busy time alone saturates
        // before the link does), else the copy stream's busy fraction
        bool room;
        if (cfg->link_gbs > 0.f && obs->interval_ns > 0) {
            const double gbs = (double)obs->copy_bytes / (double)obs->interval_ns;  // bytes per ns = GB/s
            room = gbs < (double)cfg->copy_busy_max * (double)cfg->link_gbs;
        } else {
            room = obs->copy_busy < cfg->copy_busy_max;
        }
        const bool want_grow = miss_rate > cfg->miss_grow && room;
        const bool want_shrink = obs->ready_misses == 0 && obs->ring_occupancy < cfg->occupancy_shrink;
        st.grow_run = want_grow ? prev->grow_run + 1 : 0;
        st.shrink_run = want_shrink ? prev->shrink_run + 1 : 0;
        ring = clamp_u32(prev->ring_slots, lo, hi);
        reason = ring != prev->ring_slots ? KVS_POLICY_CLAMP : KVS_POLICY_HOLD;
        // a change that a bound leaves without effect keeps its run counting
        if (st.grow_run >= cfg->hold_steps && ring < hi) {
            ring = clamp_u32((uint64_t)ring + cfg->step_slots, lo, hi);
            reason = KVS_POLICY_GROW;
            st.grow_run = st.shrink_run = 0;
        } else if (st.shrink_run >= cfg->hold_steps && ring > lo) {
            ring = clamp_u32(ring > cfg->step_slots ? ring - cfg->step_slots : 0, lo, hi);
            reason = KVS_POLICY_SHRINK;
            st.grow_run = st.shrink_run = 0;
        }
    }
    st.ring_slots = ring;

    kvs_policy_decision d;
    d.ring_slots = ring;
    d.resident_slots = cfg->budget_slots - ring;
    const uint64_t per_layer = d.resident_slots / cfg->n_layers;
    d.resident_pages_per_layer = ppl < per_layer ? ppl : per_layer;
    d.pages_per_layer = ppl;
    d.reason = reason;
    d.changed = ring != prev->ring_slots;
    *next = st;
    *out = d;
    return KVS_OK;
}
