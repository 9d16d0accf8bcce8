// Decode-step runtime: a stack of MoE layers with a pre-norm residual,
// h_{l+1} = h_l + MoE_l(RMSNorm(h_l)).
//
// Per layer with a host-managed pool (page 4's cache flow, page 1 section 3): router ->
// routed ids to the host -> slot-pool ensure (misses start uploading on the copy stream) ->
// FFN over the experts that were already resident while the misses upload -> wait for the
// uploads -> FFN over the missed experts -> release the slots -> combine with the residual
// (and the shared experts, page 3: always-resident experts outside the pool) and the next
// layer's RMSNorm.  With a device-managed pool the LRU runs on the GPU (moe_cache_plan) and
// the GEMVs fill the missed slots themselves; with every expert resident the FFN reads the
// resident pool.  Neither of those needs the host during a step, so a whole step can be
// captured once as a CUDA graph and replayed.
#include <algorithm>
#include <chrono>
#include <vector>

#include "moe_common.cuh"

namespace {

inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct StackWs {
    size_t ids, w, partial, table, hit, miss, hA, hB, xn, ids_s, w_s, partial_s, tmp, fill, gin, gout, nact,
        pf_ids, pf_w, pf_table, pf_fill, ffn, total;
    size_t ffn_bytes;
};

StackWs stack_ws(int H, int F, int qtype, int E, int k, int T, int n_shared) {
    StackWs L;
    size_t off = 0;
    L.ids = off;       off = align256(off + (size_t)T * k * 4);
    L.w = off;         off = align256(off + (size_t)T * k * 4);
    L.partial = off;   off = align256(off + (size_t)T * k * H * 4);
    L.table = off;     off = align256(off + (size_t)E * 4);
    L.hit = off;       off = align256(off + (size_t)E * 4);
    L.miss = off;      off = align256(off + (size_t)E * 4);
    L.hA = off;        off = align256(off + (size_t)T * H * 4);
    L.hB = off;        off = align256(off + (size_t)T * H * 4);
    L.xn = off;        off = align256(off + (size_t)T * H * 4);
    const int ns = n_shared > 0 ? n_shared : 0;
    L.ids_s = off;     off = align256(off + (size_t)T * ns * 4);
    L.w_s = off;       off = align256(off + (size_t)T * ns * 4);
    L.partial_s = off; off = align256(off + (size_t)T * ns * H * 4);
    L.tmp = off;       off = align256(off + (size_t)T * H * 4);
    L.fill = off;      off = align256(off + (size_t)E * 8);
    L.gin = off;       off = align256(off + (size_t)T * H * 4);
    L.gout = off;      off = align256(off + (size_t)T * H * 4);
    L.nact = off;      off = align256(off + 8);
    L.pf_ids = off;    off = align256(off + 2 * (size_t)T * k * 4);   // predicted ids, depth 1 and 2
    L.pf_w = off;      off = align256(off + 2 * (size_t)T * k * 4);
    L.pf_table = off;  off = align256(off + 2 * (size_t)E * 4);
    L.pf_fill = off;   off = align256(off + 2 * (size_t)E * 8);
    // the FFN workspace of a call depends on its token count (the gate/up K split is chosen per
    // count), and not monotonically: size it for every batch up to T
    size_t f = 0;
    for (int t = 1; t <= T; ++t) {
        f = std::max(f, moe_decode_workspace_bytes(t, H, F, qtype, E, k));
        if (ns > 0) f = std::max(f, moe_decode_workspace_bytes(t, H, F, qtype, ns, ns));
    }
    L.ffn = off;       off = align256(off + f);
    L.ffn_bytes = f;
    L.total = off;
    return L;
}

struct EventPair {
    cudaEvent_t a, b;
};

}  // namespace

struct moe_stack {
    moe_stack_desc d{};
    StackWs L{};
    std::vector<const uint16_t *> w_router;
    std::vector<const float *> bias;
    std::vector<moe_cache *> caches;
    std::vector<int> group_of_layer;   // -1: resident
    std::vector<int> group_first, group_n;
    int32_t *ids_h = nullptr;          // pinned [max_T * k]
    int32_t *slots_h = nullptr;
    cudaEvent_t ids_ready = nullptr;
    cudaStream_t last_stream = nullptr;
    // profiling
    std::vector<cudaEvent_t> ev_pool;
    size_t ev_used = 0;
    std::vector<std::pair<int, EventPair>> timed;  // (kind, events)
    moe_stack_profile prof{};
    char *ws = nullptr;
    // CUDA graphs of whole decode steps, per batch size (device-managed stacks)
    cudaStream_t cap_stream = nullptr;                  // graphs are captured here (never the
                                                        // legacy default stream), launched on the caller's
    cudaGraphExec_t graph[MOE_DECODE_MAX_T + 1] = {};
    uint64_t graph_launches[MOE_DECODE_MAX_T + 1] = {};  // kernels per captured step
    bool eager_done[MOE_DECODE_MAX_T + 1] = {};
    uint64_t nact_pending = 0;  // routed FFN calls counted on the device since the last harvest
    // cross-layer prefetch: side stream and the events ordering it against the layer's stream
    cudaStream_t pf_stream = nullptr;
    cudaEvent_t pf_fork = nullptr, pf_rdone = nullptr, pf_pdone = nullptr, pf_fdone = nullptr;
    bool pf_pending = false;  // side work forked by the previous layer not yet joined
};

namespace {

enum { K_ROUTER = 0, K_PERMUTE, K_GATEUP, K_DOWN, K_COMBINE };

int get_event(moe_stack *st, cudaEvent_t *out) {
    if (st->ev_used == st->ev_pool.size()) {
        cudaEvent_t e;
        MOE_TRY_CUDA(cudaEventCreate(&e));
        st->ev_pool.push_back(e);
    }
    *out = st->ev_pool[st->ev_used++];
    return MOE_OK;
}

// Profiling: adds the active-expert count the permute kernel left in the FFN workspace to a
// device-side sum (for the byte accounting of layers whose routing the host never sees).
__global__ void nact_add_kernel(const int32_t *n_active, unsigned long long *sum) {
    if (threadIdx.x == 0) *sum += (unsigned long long)*n_active;
}

// Accumulates the elapsed times of recorded event pairs (all complete) and recycles them.
int harvest(moe_stack *st) {
    if (st->nact_pending) {  // routed FFN calls whose active experts were counted on the device
        unsigned long long sum = 0;
        MOE_TRY_CUDA(cudaMemcpy(&sum, st->ws + st->L.nact, 8, cudaMemcpyDeviceToHost));
        MOE_TRY_CUDA(cudaMemset(st->ws + st->L.nact, 0, 8));
        st->prof.gateup_bytes += (double)sum * 2 * moe_matrix_bytes(st->d.qtype, st->d.F, st->d.H);
        st->prof.down_bytes += (double)sum * moe_matrix_bytes(st->d.qtype, st->d.H, st->d.F);
        st->nact_pending = 0;
    }
    for (auto &te : st->timed) {
        float ms = 0.f;
        MOE_TRY_CUDA(cudaEventElapsedTime(&ms, te.second.a, te.second.b));
        switch (te.first) {
            case K_ROUTER: st->prof.router_ms += ms; break;
            case K_PERMUTE: st->prof.permute_ms += ms; break;
            case K_GATEUP: st->prof.gateup_ms += ms; break;
            case K_DOWN: st->prof.down_ms += ms; break;
            default: st->prof.combine_ms += ms; break;
        }
    }
    st->timed.clear();
    st->ev_used = 0;
    return MOE_OK;
}

int begin_timed(moe_stack *st, cudaStream_t s, EventPair *ep) {
    if (st->d.profile < 2) return MOE_OK;
    int rc = get_event(st, &ep->a);
    if (rc) return rc;
    rc = get_event(st, &ep->b);
    if (rc) return rc;
    MOE_TRY_CUDA(cudaEventRecord(ep->a, s));
    return MOE_OK;
}

int end_timed(moe_stack *st, cudaStream_t s, int kind, EventPair ep) {
    if (st->d.profile < 2) return MOE_OK;
    MOE_TRY_CUDA(cudaEventRecord(ep.b, s));
    st->timed.push_back({kind, ep});
    return MOE_OK;
}

// One FFN call with per-kernel timing when profiling.
int ffn_call(moe_stack *st, const float *x, int T, int E, int k, const int32_t *ids, const float *w,
             const int32_t *table, int n_slots, const void *pool, const int32_t *subset, int n_subset,
             float *partial, int n_active, cudaStream_t s, const uint64_t *fill = nullptr) {
    const moe_stack_desc &d = st->d;
    moe_ffn_timing tm{};
    const moe_ffn_timing *tp = nullptr;
    if (d.profile >= 1) {
        int rc;
        if ((rc = get_event(st, &tm.gateup0)) || (rc = get_event(st, &tm.gateup1))) return rc;
        if (d.profile >= 2)
            if ((rc = get_event(st, &tm.permute0)) || (rc = get_event(st, &tm.permute1)) ||
                (rc = get_event(st, &tm.down0)) || (rc = get_event(st, &tm.down1)))
                return rc;
        tp = &tm;
    }
    const int rc = moe_expert_ffn_core(x, MOE_F32, T, d.H, d.F, d.qtype, E, k, ids, w, table, n_slots,
                                       pool, d.slot_bytes, subset, n_subset, fill, partial,
                                       st->ws + st->L.ffn, st->L.ffn_bytes, s, tp);
    if (rc) return rc;
    st->prof.kernel_launches += moe_decode_ffn_launches(T, d.H, d.F, d.qtype, E, k);
    if (d.profile >= 1) {
        st->timed.push_back({K_GATEUP, {tm.gateup0, tm.gateup1}});
        if (d.profile >= 2) {
            st->timed.push_back({K_PERMUTE, {tm.permute0, tm.permute1}});
            st->timed.push_back({K_DOWN, {tm.down0, tm.down1}});
        }
        st->prof.gateup_launches++;
        st->prof.down_launches++;
    }
    if (d.profile >= 1 && n_active >= 0) {
        st->prof.gateup_bytes += (double)n_active * 2 * moe_matrix_bytes(d.qtype, d.F, d.H);
        st->prof.down_bytes += (double)n_active * moe_matrix_bytes(d.qtype, d.H, d.F);
    } else if (d.profile >= 1) {  // not known on the host: count on the device (after the GEMVs)
        nact_add_kernel<<<1, 32, 0, s>>>((const int32_t *)(st->ws + st->L.ffn),
                                         (unsigned long long *)(st->ws + st->L.nact));
        MOE_TRY_CUDA(cudaGetLastError());
        ++st->nact_pending;
    }
    return MOE_OK;
}

// RMSNorm epsilon of the stack's pre-norm
#define MOE_STACK_EPS 1e-6f

// Cross-layer speculative prefetch (page 3, tiered MoE scheduling note, section 2.3: while the
// GPU computes the current layer a second stream prefetches the experts the next one or two
// layers will use; section 4.3: depth 2).  After layer `layer`'s plan: the routers of the next
// `prefetch_depth` layers are applied to this layer's input x (their prediction), their pools
// plan the predicted ids speculatively, and the predicted misses are copied into their slots —
// all on the side stream, ordered by events: the main stream waits for the routers before x
// is overwritten (the combine), for the plans before the next plan, for the copies before the
// next FFN.
int prefetch_fork(moe_stack *st, int layer, const float *x, int T, cudaStream_t s) {
    const moe_stack_desc &d = st->d;
    const StackWs &L = st->L;
    int targets[2], n = 0;
    for (int dd = 1; dd <= d.prefetch_depth && dd <= 2; ++dd) {
        const int l2 = layer + dd;
        if (l2 < d.n_layers && st->group_of_layer[l2] >= 0) targets[n++] = l2;
    }
    if (n == 0) return MOE_OK;
    if (!st->pf_stream) {
        MOE_TRY_CUDA(cudaStreamCreateWithFlags(&st->pf_stream, cudaStreamNonBlocking));
        for (cudaEvent_t *e : {&st->pf_fork, &st->pf_rdone, &st->pf_pdone, &st->pf_fdone})
            MOE_TRY_CUDA(cudaEventCreateWithFlags(e, cudaEventDisableTiming));
    }
    cudaStream_t ps = st->pf_stream;
    const size_t R = (size_t)T * d.k;
    int32_t *pids = (int32_t *)(st->ws + L.pf_ids);
    float *pw = (float *)(st->ws + L.pf_w);
    int32_t *ptab = (int32_t *)(st->ws + L.pf_table);
    uint64_t *pfill = (uint64_t *)(st->ws + L.pf_fill);
    MOE_TRY_CUDA(cudaEventRecord(st->pf_fork, s));
    MOE_TRY_CUDA(cudaStreamWaitEvent(ps, st->pf_fork, 0));
    int rc;
    for (int i = 0; i < n; ++i)
        if ((rc = moe_router_topk_threshold(x, MOE_F32, T, d.H, st->w_router[targets[i]], st->bias[targets[i]], d.E,
                                            d.k, d.load_threshold, pids + i * R, pw + i * R, nullptr,
                                            (moe_stream_t)ps)))
            return rc;
    MOE_TRY_CUDA(cudaEventRecord(st->pf_rdone, ps));
    for (int i = 0; i < n; ++i)
        if ((rc = moe_cache_prefetch_plan(st->caches[st->group_of_layer[targets[i]]], targets[i], pids + i * R, T,
                                          d.k, ptab + i * d.E, pfill + i * d.E, (moe_stream_t)ps)))
            return rc;
    MOE_TRY_CUDA(cudaEventRecord(st->pf_pdone, ps));
    for (int i = 0; i < n; ++i)
        if ((rc = moe_cache_prefetch_fill(st->caches[st->group_of_layer[targets[i]]], ptab + i * d.E,
                                          pfill + i * d.E, (moe_stream_t)ps)))
            return rc;
    MOE_TRY_CUDA(cudaEventRecord(st->pf_fdone, ps));
    st->prof.kernel_launches += 3 * n;
    st->pf_pending = true;
    return MOE_OK;
}

// One layer: y = h + MoE(RMSNorm(h)).  norm_in: compute RMSNorm(h) here (else the previous
// layer's combine left it in the xn buffer); norm_out: leave RMSNorm(y) in xn for the next.
int layer_step(moe_stack *st, int layer, const float *h, float *y, int T, int32_t *ids_out,
               float *w_out, cudaStream_t s, bool norm_in, bool norm_out) {
    const moe_stack_desc &d = st->d;
    const StackWs &L = st->L;
    int32_t *ids_d = (int32_t *)(st->ws + L.ids);
    float *w_d = (float *)(st->ws + L.w);
    float *partial = (float *)(st->ws + L.partial);
    int32_t *table = (int32_t *)(st->ws + L.table);
    int32_t *hit_d = (int32_t *)(st->ws + L.hit);
    int32_t *miss_d = (int32_t *)(st->ws + L.miss);
    float *x = (float *)(st->ws + L.xn);
    int rc;
    EventPair ep{};

    if (norm_in) {
        if ((rc = moe_combine_rmsnorm(nullptr, T, 0, d.H, h, nullptr, x, MOE_STACK_EPS, (moe_stream_t)s)))
            return rc;
        st->prof.kernel_launches += 1;
    }
    if ((rc = begin_timed(st, s, &ep))) return rc;
    if ((rc = moe_router_topk_threshold(x, MOE_F32, T, d.H, st->w_router[layer], st->bias[layer], d.E, d.k,
                                        d.load_threshold, ids_d, w_d, nullptr, (moe_stream_t)s)))
        return rc;
    st->prof.kernel_launches += 1;
    if ((rc = end_timed(st, s, K_ROUTER, ep))) return rc;

    const int g = st->group_of_layer[layer];
    bool forked = false;
    if (g >= 0 && d.device_managed) {
        // the pool's bookkeeping on the GPU, then the FFN filling the missed experts' slots
        moe_cache *c = st->caches[g];
        uint64_t *fill = (uint64_t *)(st->ws + L.fill);
        // the previous layer's speculative plans come before this plan
        if (st->pf_pending) MOE_TRY_CUDA(cudaStreamWaitEvent(s, st->pf_pdone, 0));
        if ((rc = moe_cache_plan(c, layer, ids_d, T, d.k, table, fill, (moe_stream_t)s))) return rc;
        st->prof.kernel_launches += 1;
        if (st->pf_pending) {  // and its copies land before this FFN reads the slots
            MOE_TRY_CUDA(cudaStreamWaitEvent(s, st->pf_fdone, 0));
            st->pf_pending = false;
        }
        if (d.prefetch_depth > 0) {
            if ((rc = prefetch_fork(st, layer, x, T, s))) return rc;
            forked = st->pf_pending;
        }
        int ns = 0;
        const void *pool = moe_cache_pool(c, &ns);
        if ((rc = ffn_call(st, x, T, d.E, d.k, ids_d, w_d, table, ns, pool, nullptr, 0, partial, -1, s, fill)))
            return rc;
    } else if (g >= 0) {
        moe_cache *c = st->caches[g];
        MOE_TRY_CUDA(cudaMemcpyAsync(st->ids_h, ids_d, (size_t)T * d.k * 4, cudaMemcpyDeviceToHost, s));
        MOE_TRY_CUDA(cudaEventRecord(st->ids_ready, s));
        const auto w0 = std::chrono::steady_clock::now();
        MOE_TRY_CUDA(cudaEventSynchronize(st->ids_ready));
        st->prof.host_wait_ms +=
            std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - w0).count();
        if (d.profile && (rc = harvest(st))) return rc;  // everything recorded so far has completed
        int n_miss = 0;
        uint8_t miss_mask[MOE_MAX_E];
        if ((rc = moe_cache_ensure(c, layer, st->ids_h, T, d.k, st->slots_h, &n_miss, miss_mask,
                                   nullptr, (moe_stream_t)s)))
            return rc;
        bool want[MOE_MAX_E] = {false};
        for (int i = 0; i < T * d.k; ++i)
            if (st->ids_h[i] >= 0) want[st->ids_h[i]] = true;  // -1: a dropped route
        int32_t hits[MOE_MAX_E], misses[MOE_MAX_E], tbl[MOE_MAX_E];
        uint64_t fsrc[MOE_MAX_E];
        int nh = 0, nm = 0;
        bool any_bypass = false;
        for (int e = 0; e < d.E; ++e) {
            tbl[e] = moe_cache_lookup(c, layer, e);
            fsrc[e] = 0ull;
            if (!want[e]) continue;
            if (miss_mask[e]) {
                misses[nm++] = e;
            } else {
                hits[nh++] = e;  // resident, or bypassed by the admission policy (no slot):
                if (tbl[e] < 0) {  // then read from its pinned host image
                    fsrc[e] = (uint64_t)(uintptr_t)moe_cache_image(c, layer, e);
                    any_bypass = true;
                }
            }
        }
        uint64_t *fill = any_bypass ? (uint64_t *)(st->ws + L.fill) : nullptr;
        if (fill) {  // the u64 table as two runs of 32-bit words
            int32_t *dst[3] = {(int32_t *)fill, (int32_t *)fill + d.E, nullptr};
            const int n[3] = {d.E, d.E, 0};
            const int32_t *src[3] = {(const int32_t *)fsrc, (const int32_t *)fsrc + d.E, nullptr};
            if ((rc = moe_write_ints(dst, n, src, s))) return rc;
            st->prof.kernel_launches += 1;
        }
        const bool two_phase = d.overlap && nh > 0 && nm > 0;
        {
            int32_t *dst[3] = {table, hit_d, miss_d};
            const int n[3] = {d.E, two_phase ? nh : 0, two_phase ? nm : 0};
            const int32_t *src[3] = {tbl, hits, misses};
            if ((rc = moe_write_ints(dst, n, src, s))) return rc;
            st->prof.kernel_launches += 1;
            st->prof.h2d_copies += n_miss;
        }
        {
            int ns = 0;
            const void *pool = moe_cache_pool(c, &ns);
            if (two_phase) {
                if ((rc = ffn_call(st, x, T, d.E, d.k, ids_d, w_d, table, ns, pool, hit_d, nh, partial, nh, s,
                                   fill)))
                    return rc;
                if ((rc = moe_cache_wait_uploads(c, (moe_stream_t)s))) return rc;
                if ((rc = ffn_call(st, x, T, d.E, d.k, ids_d, w_d, table, ns, pool, miss_d, nm, partial, nm, s)))
                    return rc;
            } else {
                if ((rc = moe_cache_wait_uploads(c, (moe_stream_t)s))) return rc;
                if ((rc = ffn_call(st, x, T, d.E, d.k, ids_d, w_d, table, ns, pool, nullptr, 0, partial,
                                   nh + nm, s, fill)))
                    return rc;
            }
        }
        if ((rc = moe_cache_release(c, (moe_stream_t)s))) return rc;
    } else {
        const void *pool = (const char *)d.resident_pool + (size_t)layer * d.E * d.slot_bytes;
        if ((rc = ffn_call(st, x, T, d.E, d.k, ids_d, w_d, nullptr, d.E, pool, nullptr, 0, partial, -1, s)))
            return rc;
    }

    const float *extra = h;
    if (d.n_shared > 0) {
        const void *spool = (const char *)d.shared_pool + (size_t)layer * d.n_shared * d.slot_bytes;
        int32_t *ids_s = (int32_t *)(st->ws + L.ids_s);
        float *w_s = (float *)(st->ws + L.w_s);
        float *partial_s = (float *)(st->ws + L.partial_s);
        float *tmp = (float *)(st->ws + L.tmp);
        if ((rc = ffn_call(st, x, T, d.n_shared, d.n_shared, ids_s, w_s, nullptr, d.n_shared, spool,
                           nullptr, 0, partial_s, d.n_shared, s)))
            return rc;
        if ((rc = begin_timed(st, s, &ep))) return rc;
        if ((rc = moe_combine(partial_s, T, d.n_shared, d.H, h, tmp, (moe_stream_t)s))) return rc;
        st->prof.kernel_launches += 1;
        if ((rc = end_timed(st, s, K_COMBINE, ep))) return rc;
        extra = tmp;
    }
    if (forked) MOE_TRY_CUDA(cudaStreamWaitEvent(s, st->pf_rdone, 0));  // the predictions read x
    if ((rc = begin_timed(st, s, &ep))) return rc;
    if ((rc = moe_combine_rmsnorm_routes(partial, d.load_threshold > 0.f ? ids_d : nullptr, T, d.k, d.H, extra, y,
                                         norm_out ? x : nullptr, MOE_STACK_EPS, s)))
        return rc;
    st->prof.kernel_launches += 1;
    if ((rc = end_timed(st, s, K_COMBINE, ep))) return rc;

    if (ids_out) MOE_TRY_CUDA(cudaMemcpyAsync(ids_out, ids_d, (size_t)T * d.k * 4, cudaMemcpyDeviceToHost, s));
    if (w_out) MOE_TRY_CUDA(cudaMemcpyAsync(w_out, w_d, (size_t)T * d.k * 4, cudaMemcpyDeviceToHost, s));
    st->prof.layers++;
    return MOE_OK;
}

}  // namespace

extern "C" int moe_stack_workspace(int H, int F, int qtype, int E, int k, int max_T, int n_shared,
                                   size_t *bytes) {
    MOE_CHECK(bytes && H > 0 && F > 0 && H % 32 == 0 && F % 32 == 0);
    MOE_CHECK(qtype == MOE_Q8_0 || qtype == MOE_Q4_SM);
    MOE_CHECK(E >= 1 && E <= MOE_MAX_E && k >= 1 && k <= MOE_MAX_K && k <= E);
    MOE_CHECK(max_T >= 1 && max_T <= MOE_DECODE_MAX_T && n_shared >= 0 && n_shared <= MOE_MAX_K);
    *bytes = stack_ws(H, F, qtype, E, k, max_T, n_shared).total;
    return MOE_OK;
}

extern "C" int moe_stack_create(const moe_stack_desc *desc, moe_stack **out) {
    MOE_CHECK(desc && out);
    *out = nullptr;
    const moe_stack_desc &d = *desc;
    size_t need = 0;
    int rc = moe_stack_workspace(d.H, d.F, d.qtype, d.E, d.k, d.max_T, d.n_shared, &need);
    if (rc) return rc;
    MOE_CHECK(d.n_layers >= 1 && d.w_router);
    MOE_CHECK(d.workspace && ((uintptr_t)d.workspace % 256) == 0 && d.ws_bytes >= need);
    MOE_CHECK(d.slot_bytes >= moe_expert_image_bytes(d.qtype, d.H, d.F) && d.slot_bytes % 256 == 0);
    MOE_CHECK(d.n_groups >= 0);
    if (d.n_groups == 0) MOE_CHECK(d.resident_pool != nullptr);
    else MOE_CHECK(d.caches != nullptr);
    if (d.n_shared > 0) MOE_CHECK(d.shared_pool != nullptr);
    MOE_CHECK(d.prefetch_depth >= 0 && d.prefetch_depth <= 2);
    MOE_CHECK(d.load_threshold >= 0.f && d.load_threshold <= 1.f);
    if (d.prefetch_depth > 0 && !(d.device_managed && d.n_groups > 0)) return MOE_ERR_UNSUPPORTED;

    moe_stack *st = new moe_stack();
    st->d = d;
    st->L = stack_ws(d.H, d.F, d.qtype, d.E, d.k, d.max_T, d.n_shared);
    st->ws = (char *)d.workspace;
    st->w_router.assign(d.w_router, d.w_router + d.n_layers);
    st->bias.assign(d.n_layers, nullptr);
    if (d.bias) st->bias.assign(d.bias, d.bias + d.n_layers);
    st->group_of_layer.assign(d.n_layers, -1);
    for (int g = 0; g < d.n_groups; ++g) {
        moe_cache *c = d.caches[g];
        int first = 0, n = 0;
        if (!c || moe_cache_layer_range(c, &first, &n) != MOE_OK || first + n > d.n_layers) {
            delete st;
            return MOE_ERR_INVALID;
        }
        if (moe_cache_is_device_managed(c) != (d.device_managed != 0)) {
            delete st;
            return MOE_ERR_INVALID;  // the caches' kind must match the stack's
        }
        st->caches.push_back(c);
        for (int l = first; l < first + n; ++l) st->group_of_layer[l] = g;
    }
    if (d.n_groups > 0)
        for (int l = 0; l < d.n_layers; ++l)
            if (st->group_of_layer[l] < 0) {
                delete st;
                return MOE_ERR_INVALID;  // every layer must belong to a group
            }
    if (cudaMemset(st->ws + st->L.nact, 0, 8) != cudaSuccess ||
        cudaHostAlloc(&st->ids_h, (size_t)d.max_T * d.k * 4, cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc(&st->slots_h, (size_t)d.max_T * d.k * 4, cudaHostAllocDefault) != cudaSuccess ||
        cudaEventCreateWithFlags(&st->ids_ready, cudaEventDisableTiming) != cudaSuccess) {
        moe_stack_destroy(st);
        return MOE_ERR_CUDA;
    }
    if (d.n_shared > 0) {
        // constant routing of the shared experts: every token, every shared expert, weight 1
        std::vector<int32_t> ids((size_t)d.max_T * d.n_shared);
        std::vector<float> w((size_t)d.max_T * d.n_shared, 1.0f);
        for (int t = 0; t < d.max_T; ++t)
            for (int j = 0; j < d.n_shared; ++j) ids[(size_t)t * d.n_shared + j] = j;
        if (cudaMemcpy(st->ws + st->L.ids_s, ids.data(), ids.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemcpy(st->ws + st->L.w_s, w.data(), w.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess) {
            moe_stack_destroy(st);
            return MOE_ERR_CUDA;
        }
    }
    *out = st;
    return MOE_OK;
}

extern "C" int moe_stack_layer(moe_stack *st, int layer, const float *x_in, float *y_out, int T,
                               int32_t *ids_host_out, float *weights_host_out, moe_stream_t s) {
    MOE_CHECK(st && x_in && y_out);
    MOE_CHECK(layer >= 0 && layer < st->d.n_layers);
    MOE_CHECK(T >= 1 && T <= st->d.max_T);
    cudaStream_t cs = moe_cuda_stream(s);
    st->last_stream = cs;
    const int rc = layer_step(st, layer, x_in, y_out, T, ids_host_out, weights_host_out, cs, true, false);
    if (rc == MOE_OK && st->pf_pending) {  // a single layer leaves no work behind on the side stream
        MOE_TRY_CUDA(cudaStreamWaitEvent(cs, st->pf_fdone, 0));
        st->pf_pending = false;
    }
    return rc;
}

namespace {

int run_step(moe_stack *st, const float *x_in, float *y_out, int T, int32_t *ids_host_out,
             float *weights_host_out, cudaStream_t cs) {
    const int L = st->d.n_layers;
    float *hA = (float *)(st->ws + st->L.hA), *hB = (float *)(st->ws + st->L.hB);
    const float *cur = x_in;
    const size_t per = (size_t)T * st->d.k;
    for (int l = 0; l < L; ++l) {
        float *out = (l == L - 1) ? y_out : ((l & 1) ? hB : hA);
        const int rc = layer_step(st, l, cur, out, T, ids_host_out ? ids_host_out + l * per : nullptr,
                                  weights_host_out ? weights_host_out + l * per : nullptr, cs, l == 0,
                                  l + 1 < L);
        if (rc) return rc;
        cur = out;
    }
    if (st->pf_pending) {  // every side-stream copy joins the step
        MOE_TRY_CUDA(cudaStreamWaitEvent(cs, st->pf_fdone, 0));
        st->pf_pending = false;
    }
    return MOE_OK;
}

// Captures one whole step (device-managed stacks) reading gin and writing gout, on the
// stack's own capture stream (nothing executes during a capture).
int capture_step(moe_stack *st, int T) {
    float *gin = (float *)(st->ws + st->L.gin), *gout = (float *)(st->ws + st->L.gout);
    const uint64_t launches0 = st->prof.kernel_launches;
    if (!st->cap_stream) MOE_TRY_CUDA(cudaStreamCreateWithFlags(&st->cap_stream, cudaStreamNonBlocking));
    cudaStream_t cs = st->cap_stream;
    MOE_TRY_CUDA(cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed));
    const int rc = run_step(st, gin, gout, T, nullptr, nullptr, cs);
    cudaGraph_t graph = nullptr;
    const cudaError_t ec = cudaStreamEndCapture(cs, &graph);
    st->graph_launches[T] = st->prof.kernel_launches - launches0;
    st->prof.kernel_launches = launches0;
    if (rc != MOE_OK) {
        if (graph) cudaGraphDestroy(graph);
        return rc;
    }
    if (ec != cudaSuccess) return MOE_ERR_CUDA;
    const cudaError_t ei = cudaGraphInstantiate(&st->graph[T], graph, 0);
    cudaGraphDestroy(graph);
    if (ei != cudaSuccess) {
        st->graph[T] = nullptr;
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

}  // namespace

extern "C" int moe_stack_decode(moe_stack *st, const float *x_in, float *y_out, int T,
                                int32_t *ids_host_out, float *weights_host_out, moe_stream_t s) {
    MOE_CHECK(st && x_in && y_out);
    MOE_CHECK(T >= 1 && T <= st->d.max_T);
    cudaStream_t cs = moe_cuda_stream(s);
    st->last_stream = cs;
    const moe_stack_desc &d = st->d;
    const bool host_free = d.device_managed || d.n_groups == 0;  // no host round trip inside a step
    const bool graphable = d.use_graph && host_free && !d.profile && !ids_host_out && !weights_host_out;
    if (graphable && st->eager_done[T]) {
        if (!st->graph[T]) {
            const int rc = capture_step(st, T);
            if (rc) return rc;
        }
        const size_t bytes = (size_t)T * d.H * 4;
        MOE_TRY_CUDA(cudaMemcpyAsync(st->ws + st->L.gin, x_in, bytes, cudaMemcpyDeviceToDevice, cs));
        MOE_TRY_CUDA(cudaGraphLaunch(st->graph[T], cs));
        MOE_TRY_CUDA(cudaMemcpyAsync(y_out, st->ws + st->L.gout, bytes, cudaMemcpyDeviceToDevice, cs));
        st->prof.kernel_launches += st->graph_launches[T];
        st->prof.layers += d.n_layers;
        st->prof.steps++;
        return MOE_OK;
    }
    // eager: every launch issued now (the first call of a graph-captured stack runs eagerly so
    // that one-time set-up never happens inside a capture)
    const int rc = run_step(st, x_in, y_out, T, ids_host_out, weights_host_out, cs);
    if (rc) return rc;
    st->eager_done[T] = true;
    st->prof.steps++;
    return MOE_OK;
}

extern "C" int moe_stack_profile_get(moe_stack *st, moe_stack_profile *out) {
    MOE_CHECK(st && out);
    if (st->last_stream) MOE_TRY_CUDA(cudaStreamSynchronize(st->last_stream));
    const int rc = harvest(st);
    if (rc) return rc;
    *out = st->prof;
    return MOE_OK;
}

extern "C" int moe_stack_profile_reset(moe_stack *st) {
    MOE_CHECK(st);
    if (st->last_stream) MOE_TRY_CUDA(cudaStreamSynchronize(st->last_stream));
    st->timed.clear();
    st->ev_used = 0;
    st->prof = moe_stack_profile{};
    st->nact_pending = 0;
    MOE_TRY_CUDA(cudaMemset(st->ws + st->L.nact, 0, 8));
    return MOE_OK;
}

extern "C" int moe_stack_set_profile(moe_stack *st, int level) {
    MOE_CHECK(st && level >= 0 && level <= 2);
    if (st->last_stream) MOE_TRY_CUDA(cudaStreamSynchronize(st->last_stream));
    const int rc = harvest(st);
    if (rc) return rc;
    st->d.profile = level;
    return MOE_OK;
}

namespace {
// A GPU spacer: one warp spinning for about `ns` nanoseconds of wall time (bounded), so that
// the host has queued every timed launch before the first of them can start.
__global__ void spacer_kernel(unsigned long long ns) {
    unsigned long long t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    do {
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    } while (t - t0 < ns);
}
}  // namespace

extern "C" int moe_stack_gemv_timing(moe_stack *st, const float *x_in, int T, int reps, moe_gemv_timing *out,
                                     moe_stream_t sv) {
    MOE_CHECK(st && x_in && out && reps >= 1);
    MOE_CHECK(T >= 1 && T <= st->d.max_T && T <= MOE_DECODE_MAX_T);
    const moe_stack_desc &d = st->d;
    if (d.n_groups != 0 || !d.resident_pool) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = moe_cuda_stream(sv);
    const int L = d.n_layers, R = T * d.k;
    const size_t wsb = moe_decode_workspace_bytes(T, d.H, d.F, d.qtype, d.E, d.k);
    const size_t per = align256((size_t)R * 4) * 2 + align256((size_t)R * d.H * 4) + align256(wsb);
    char *buf = nullptr;
    MOE_TRY_CUDA(cudaMalloc(&buf, per * L));
    cudaEvent_t ev[5] = {};
    int rc = MOE_OK;
    auto lay = [&](int l, int32_t **ids, float **w, float **partial, void **ws) {
        char *b = buf + per * l;
        *ids = (int32_t *)b;
        *w = (float *)(b + align256((size_t)R * 4));
        *partial = (float *)(b + 2 * align256((size_t)R * 4));
        *ws = b + 2 * align256((size_t)R * 4) + align256((size_t)R * d.H * 4);
    };
    auto stage = [&](int l, int what) {
        int32_t *ids; float *w, *partial; void *ws;
        lay(l, &ids, &w, &partial, &ws);
        const void *pool = (const char *)d.resident_pool + (size_t)l * d.E * d.slot_bytes;
        return moe_expert_ffn_stages(x_in, MOE_F32, T, d.H, d.F, d.qtype, d.E, d.k, ids, w, nullptr, d.E, pool,
                                     d.slot_bytes, nullptr, 0, nullptr, partial, ws, wsb, s, nullptr, what);
    };
    for (int i = 0; i < 5 && rc == MOE_OK; ++i)
        if (cudaEventCreate(&ev[i]) != cudaSuccess) rc = MOE_ERR_CUDA;
    for (int l = 0; l < L && rc == MOE_OK; ++l) {  // routing of every layer, then its permute
        int32_t *ids; float *w, *partial; void *ws;
        lay(l, &ids, &w, &partial, &ws);
        rc = moe_router_topk(x_in, MOE_F32, T, d.H, st->w_router[l], st->bias[l], d.E, d.k, ids, w, nullptr, sv);
        if (rc == MOE_OK) rc = stage(l, MOE_FFN_PERMUTE);
    }
    // x_in is complete long before: the gate/up rounds may start early
    for (int l = 0; l < L && rc == MOE_OK; ++l) rc = stage(l, MOE_FFN_GATEUP | MOE_FFN_REDUCE | MOE_FFN_X_READY);
    for (int l = 0; l < L && rc == MOE_OK; ++l) rc = stage(l, MOE_FFN_DOWN);
    for (int l = 0; l < L && rc == MOE_OK; ++l) rc = stage(l, MOE_FFN_ALL);
    if (rc == MOE_OK) {  // about 40 us of host time per launch to queue, at least 2 ms
        const unsigned long long ns = std::max(2000000ull, 40000ull * 3 * (unsigned long long)reps * L);
        spacer_kernel<<<1, 32, 0, s>>>(ns);
        if (cudaGetLastError() != cudaSuccess) rc = MOE_ERR_CUDA;
    }
    if (rc == MOE_OK && cudaEventRecord(ev[0], s) != cudaSuccess) rc = MOE_ERR_CUDA;
    for (int r = 0; r < reps && rc == MOE_OK; ++r)
        for (int l = 0; l < L && rc == MOE_OK; ++l) rc = stage(l, MOE_FFN_GATEUP | MOE_FFN_X_READY);
    if (rc == MOE_OK && cudaEventRecord(ev[1], s) != cudaSuccess) rc = MOE_ERR_CUDA;
    for (int r = 0; r < reps && rc == MOE_OK; ++r)
        for (int l = 0; l < L && rc == MOE_OK; ++l) rc = stage(l, MOE_FFN_REDUCE);
    if (rc == MOE_OK && cudaEventRecord(ev[2], s) != cudaSuccess) rc = MOE_ERR_CUDA;
    for (int r = 0; r < reps && rc == MOE_OK; ++r)
        for (int l = 0; l < L && rc == MOE_OK; ++l) rc = stage(l, MOE_FFN_DOWN);
    if (rc == MOE_OK && cudaEventRecord(ev[3], s) != cudaSuccess) rc = MOE_ERR_CUDA;
    for (int r = 0; r < reps && rc == MOE_OK; ++r)
        for (int l = 0; l < L && rc == MOE_OK; ++l) rc = stage(l, MOE_FFN_ALL);
    if (rc == MOE_OK && cudaEventRecord(ev[4], s) != cudaSuccess) rc = MOE_ERR_CUDA;
    if (rc == MOE_OK && cudaStreamSynchronize(s) != cudaSuccess) rc = MOE_ERR_CUDA;
    if (rc == MOE_OK) {
        float t1 = 0.f, t2 = 0.f, t3 = 0.f, t4 = 0.f;
        cudaEventElapsedTime(&t4, ev[3], ev[4]);
        cudaEventElapsedTime(&t1, ev[0], ev[1]);
        cudaEventElapsedTime(&t3, ev[1], ev[2]);
        cudaEventElapsedTime(&t2, ev[2], ev[3]);
        double nact = 0.0;
        for (int l = 0; l < L && rc == MOE_OK; ++l) {
            int32_t n = 0;
            if (cudaMemcpy(&n, buf + per * l + 2 * align256((size_t)R * 4) + align256((size_t)R * d.H * 4), 4,
                           cudaMemcpyDeviceToHost) != cudaSuccess)
                rc = MOE_ERR_CUDA;
            nact += n;
        }
        const int n_l = reps * L;
        out->gateup_us = 1e3 * t1 / n_l;
        out->down_us = 1e3 * t2 / n_l;
        out->reduce_us = 1e3 * t3 / n_l;
        out->gemv_us = 1e3 * t4 / n_l;
        out->fused = moe_get_decode_fused();
        out->gateup_bytes = nact / L * 2 * moe_matrix_bytes(d.qtype, d.F, d.H);
        out->down_bytes = nact / L * moe_matrix_bytes(d.qtype, d.H, d.F);
        out->launches = n_l;
    }
    for (int i = 0; i < 5; ++i)
        if (ev[i]) cudaEventDestroy(ev[i]);
    cudaFree(buf);
    return rc;
}

extern "C" void moe_stack_destroy(moe_stack *st) {
    if (!st) return;
    if (st->last_stream) cudaStreamSynchronize(st->last_stream);
    for (cudaEvent_t e : st->ev_pool) cudaEventDestroy(e);
    for (int t = 0; t <= MOE_DECODE_MAX_T; ++t)
        if (st->graph[t]) cudaGraphExecDestroy(st->graph[t]);
    if (st->cap_stream) cudaStreamDestroy(st->cap_stream);
    if (st->pf_stream) cudaStreamSynchronize(st->pf_stream);
    for (cudaEvent_t e : {st->pf_fork, st->pf_rdone, st->pf_pdone, st->pf_fdone})
        if (e) cudaEventDestroy(e);
    if (st->pf_stream) cudaStreamDestroy(st->pf_stream);
    if (st->ids_ready) cudaEventDestroy(st->ids_ready);
    if (st->ids_h) cudaFreeHost(st->ids_h);
    if (st->slots_h) cudaFreeHost(st->slots_h);
    delete st;
}
