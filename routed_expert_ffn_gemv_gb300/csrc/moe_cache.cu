// Expert slot pool: one per type/shape group of layers, least-recently-used.
//
// Page 4 ("llama.cpp MoE缓存实测", section "MoE缓存到底缓存了什么"): expert tensors are
// grouped by type and shape, each group gets one VRAM slot pool shared by all its
// layers, hits read VRAM, misses are uploaded, eviction is LRU.  Page 1 (section 3.2):
// the victim is the least-recently-used expert that is not part of the current request.
// Page 3: uploads come from pinned host memory with asynchronous copies.
//
// Host bookkeeping is O(log n) per hit/miss: an ordered set of (stamp, slot) gives the
// LRU order, a set of free slots gives the lowest free slot.  Every miss upload is a
// cudaMemcpyAsync on the group's copy stream, issued after the event that marks the
// slot's last reader (recorded by moe_cache_release on the compute stream).
#include <algorithm>
#include <mutex>
#include <set>
#include <utility>
#include <vector>

#include "moe_common.cuh"
#include "moe_ptx.cuh"

#define MOE_EVENT_RING 64

struct moe_cache {
    moe_cache_desc d{};
    size_t image_bytes = 0;
    std::vector<const void *> images;
    std::vector<int32_t> slot_of;     // [n_layers * E] -> slot or -1
    std::vector<int64_t> owner;       // [n_slots] -> layer_local * E + e, or -1
    std::vector<uint64_t> stamp;      // [n_slots]
    std::set<std::pair<uint64_t, int>> lru;  // occupied slots by stamp
    std::set<int> free_slots;
    uint64_t clock = 0;
    std::vector<int> last_use;        // [n_slots] -> event ring index or -1
    cudaEvent_t ring[MOE_EVENT_RING] = {};
    int ring_next = 0;
    cudaEvent_t upload_done = nullptr;
    bool upload_pending = false;
    std::vector<int> last_slots;      // slots of the last ensure (for release)
    moe_cache_stats st{};
    std::vector<uint32_t> count;      // [n_layers * E] accesses (admission policy)
    std::vector<uint64_t> last_tok;   // [n_slots] token clock at the last use (window policy)
    uint64_t tok = 0;                 // the pool's token clock
};

struct IntPayload {
    int32_t v[3][MOE_MAX_E];
};

namespace {

__global__ void write_ints_kernel(int32_t *d0, int n0, int32_t *d1, int n1, int32_t *d2, int n2,
                                  const __grid_constant__ IntPayload pay) {
    const int i = threadIdx.x;
    if (d0 && i < n0) d0[i] = pay.v[0][i];
    if (d1 && i < n1) d1[i] = pay.v[1][i];
    if (d2 && i < n2) d2[i] = pay.v[2][i];
}

void reset_state(moe_cache *c) {
    std::fill(c->slot_of.begin(), c->slot_of.end(), -1);
    std::fill(c->owner.begin(), c->owner.end(), -1);
    std::fill(c->stamp.begin(), c->stamp.end(), 0);
    std::fill(c->last_use.begin(), c->last_use.end(), -1);
    c->lru.clear();
    c->free_slots.clear();
    for (int s = 0; s < c->d.n_slots; ++s) c->free_slots.insert(s);
    c->clock = 0;
    c->upload_pending = false;
    c->last_slots.clear();
    c->st = moe_cache_stats{};
    std::fill(c->count.begin(), c->count.end(), 0u);
    std::fill(c->last_tok.begin(), c->last_tok.end(), 0ull);
    c->tok = 0;
}

// ------------------------------------------------------------------ device-managed state
//
// The recency order is an intrusive doubly linked list over the occupied slots (head =
// least recently used, tail = most recent).  Taking hits in ascending id order to the
// tail, then filling misses (ascending id) from the lowest free slot or else from the
// first list entry not owned by this request, is the same rule as the host pool's
// stamps: list order is stamp order.  Slots are only freed by a reset, so the lowest
// free slot is the fill count.

struct DevHeader {
    int32_t n_filled, head, tail, pad;
    uint64_t queries[2], hits[2], misses[2], evictions, h2d_bytes, route_queries, route_hits, ensure_calls;
    uint64_t bypassed, window_evictions;
    uint64_t pf_queries, pf_hits, pf_fills, pf_aborts;  // speculative (prefetch) requests
    uint32_t epoch, pad2;                                // real requests so far
};
static_assert(sizeof(DevHeader) <= 256, "device header");

struct DevLayout {
    size_t slot_of, owner, prev, next, img, count, recent, total;
};

DevLayout dev_layout(int n_layers, int E, int n_slots) {
    DevLayout L;
    const size_t nk = (size_t)n_layers * E;
    size_t o = 256;
    L.slot_of = o; o += (nk * 4 + 15) / 16 * 16;
    L.owner = o;   o += ((size_t)n_slots * 4 + 15) / 16 * 16;
    L.prev = o;    o += ((size_t)n_slots * 4 + 15) / 16 * 16;
    L.next = o;    o += ((size_t)n_slots * 4 + 15) / 16 * 16;
    L.img = o;     o += nk * 8;
    L.count = o;   o += (nk * 4 + 15) / 16 * 16;
    L.recent = o;  o += ((size_t)n_slots * 4 + 15) / 16 * 16;  // epoch of the last real request using a slot
    L.total = (o + 255) / 256 * 256;
    return L;
}

#define MOE_PLAN_MAX_SLOTS 12288

__global__ void __launch_bounds__(256) plan_kernel(uint8_t *__restrict__ state, DevLayout L, int ll, int E,
                                                   int n_slots, const int32_t *__restrict__ ids, int n_tokens,
                                                   int k, uint64_t image_bytes, int theta, int speculative,
                                                   int32_t *__restrict__ table_out,
                                                   uint64_t *__restrict__ src_out, int *status) {
    // Everything is read once into shared memory (one round of loads), the list is updated
    // there in parallel (one short walk from the head by one thread) and stored once.
    extern __shared__ int32_t sm[];
    int32_t *owner = sm, *prev = sm + n_slots, *next = sm + 2 * n_slots, *slot_l = sm + 3 * n_slots;
    uint32_t *cnt_l = (uint32_t *)(slot_l + E);  // accesses of the layer's experts (admission)
    unsigned char *want = (unsigned char *)(cnt_l + E), *miss = want + E;
    __shared__ int abort_flag, abort_invalid, route_hits, commit, s_head, s_tail;
    __shared__ int wsum[8];
    __shared__ int32_t vict[MOE_MAX_E], app[MOE_MAX_E];
    unsigned char *in_s = miss + E;  // hit slots (n_slots bytes)
    __shared__ int32_t s_ids[MOE_DECODE_MAX_T * MOE_MAX_K];
    __shared__ DevHeader s_hd;
    __shared__ uint64_t s_img[MOE_MAX_E];
    DevHeader *hd = (DevHeader *)state;
    int32_t *g_slot_of = (int32_t *)(state + L.slot_of);
    int32_t *g_owner = (int32_t *)(state + L.owner);
    int32_t *g_prev = (int32_t *)(state + L.prev);
    int32_t *g_next = (int32_t *)(state + L.next);
    const uint64_t *g_img = (const uint64_t *)(state + L.img);
    uint32_t *g_count = (uint32_t *)(state + L.count);
    uint32_t *g_recent = (uint32_t *)(state + L.recent);
    const int key0 = ll * E, n_ids = n_tokens * k;
    const int n_keys = (int)((L.owner - L.slot_of) / 4);  // entries the slot_of region holds
    pdl_wait();  // ids and the pool state come from earlier kernels
    pdl_trigger();
    for (int i = threadIdx.x; i < n_slots; i += blockDim.x) {
        owner[i] = g_owner[i];
        prev[i] = g_prev[i];
        next[i] = g_next[i];
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        slot_l[e] = g_slot_of[key0 + e];
        s_img[e] = g_img[key0 + e];
        cnt_l[e] = g_count[key0 + e];
        want[e] = 0;
        miss[e] = 0;
    }
    for (int i = threadIdx.x; i < n_ids; i += blockDim.x) s_ids[i] = ids[i];
    static_assert(sizeof(DevHeader) % 4 == 0, "header words");
    for (int i = threadIdx.x; i < (int)(sizeof(DevHeader) / 4); i += blockDim.x)
        ((int32_t *)&s_hd)[i] = ((const int32_t *)hd)[i];
    if (threadIdx.x == 0) {
        abort_flag = 0;
        abort_invalid = 0;
        route_hits = 0;
        commit = 0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n_ids; i += blockDim.x) {
        const int e = s_ids[i];
        if (e == -1) continue;  // a route dropped by the load threshold
        if (e < 0 || e >= E) {
            moe_set_status(status, MOE_ERR_INVALID);
            abort_flag = 1;
            abort_invalid = 1;
        } else {
            want[e] = 1;
        }
    }
    __syncthreads();
    // ---- the request: distinct experts, hits (resident) and misses, ranked by ascending id
    const int e_t = threadIdx.x;  // one expert per thread (E <= MOE_MAX_E = blockDim.x)
    const bool w_t = e_t < E && want[e_t];
    const bool hit_t = w_t && slot_l[e_t] >= 0;
    // a miss takes a slot once the expert's accesses (this one included) reach theta; before
    // that it is bypassed: read from its host image, no slot, no LRU change
    // (a speculative request admits what the real access would, but stores no access count)
    const uint32_t c_t = e_t < E ? cnt_l[e_t] + (w_t ? 1u : 0u) : 0u;
    const bool miss_any = w_t && slot_l[e_t] < 0;
    const bool miss_t = miss_any && c_t >= (uint32_t)theta, byp_t = miss_any && !miss_t;
    const int nd = __syncthreads_count(hit_t || miss_t);  // experts that need a slot
    int n_real = 0;  // routes that are not dropped
    for (int i = 0; i < n_ids; ++i) n_real += s_ids[i] != -1;
    const int nbyp = __syncthreads_count(byp_t);
    int rh = 0, rm = 0, nh = 0, nm = 0;  // this expert's rank among the hits / misses; counts
    {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        int x = (int)hit_t | ((int)miss_t << 16);
        const int v = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        int before = 0, all = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
            before += w < warp ? wsum[w] : 0;
            all += wsum[w];
        }
        const int ex = before + x - v;
        rh = ex & 0xFFFF;
        rm = ex >> 16;
        nh = all & 0xFFFF;
        nm = all >> 16;
    }
    if (threadIdx.x == 0 && !abort_flag && nd > n_slots) {
        if (!speculative) moe_set_status(status, MOE_ERR_CAPACITY);  // a prefetch just gives up
        abort_flag = 1;
    }
    if (threadIdx.x == 0) {
        s_head = s_hd.head;
        s_tail = s_hd.tail;
        if (s_head < -1 || s_head >= n_slots || s_tail < -1 || s_tail >= n_slots || s_hd.n_filled < 0 ||
            s_hd.n_filled > n_slots) {  // a corrupt header: record it, change nothing
            moe_set_status(status, MOE_ERR_CAPACITY);
            abort_flag = 1;
        }
    }
    for (int i = threadIdx.x; i < n_slots; i += blockDim.x) in_s[i] = 0;
    __syncthreads();
    if (!abort_flag) {
        // Same result as taking the hits one by one to the tail (ascending id), then for each
        // miss (ascending id) the lowest free slot, else the first list entry not owned by the
        // request, appended to the tail — done in parallel:
        // (1) unlink every hit slot: the first slot of each run of hit slots in the list joins
        //     the run's neighbours (runs touch disjoint links);
        // (a slot or link outside the pool means the state is corrupt: record it, change nothing)
        auto corrupt = [&]() {
            moe_set_status(status, MOE_ERR_CAPACITY);
            abort_flag = 1;
        };
        if (hit_t) {
            if (slot_l[e_t] < n_slots) in_s[slot_l[e_t]] = 1;
            else corrupt();
        }
        __syncthreads();
        if (hit_t && !abort_flag) {
            const int s = slot_l[e_t], pr = prev[s];
            if (pr >= n_slots) {
                corrupt();
            } else if (pr < 0 || !in_s[pr]) {
                int q = next[s], steps = 0;
                while (q >= 0 && q < n_slots && in_s[q] && steps++ <= n_slots) q = next[q];
                if (q >= n_slots || steps > n_slots) {
                    corrupt();
                } else {
                    if (pr >= 0) next[pr] = q;
                    else s_head = q;
                    if (q >= 0) prev[q] = pr;
                    else s_tail = pr;
                }
            }
        }
        __syncthreads();
        // (2) the victims: the first entries of what remains, from the head (one thread; the
        //     capacity check leaves enough entries not owned by the request);
        const int filled = s_hd.n_filled, n_free = n_slots - filled;
        const int m_evict = max(0, nm - n_free);
        if (threadIdx.x == 0 && m_evict > 0 && !abort_flag) {
            int sv = s_head;
            for (int i = 0; i < m_evict; ++i) {
                if (sv < 0 || sv >= n_slots || in_s[sv]) {
                    corrupt();
                    break;
                }
                // a prefetch never takes a slot of the last real request: that layer's kernels
                // may still be reading it (or writing it through) while the prefetch copies
                if (speculative && g_recent[sv] == s_hd.epoch && s_hd.epoch != 0u) {
                    abort_flag = 1;
                    break;
                }
                vict[i] = sv;
                sv = next[sv];
            }
            if (sv >= n_slots) corrupt();
            if (!abort_flag) {
                s_head = sv;
                if (sv >= 0) prev[sv] = -1;
                else s_tail = -1;
            }
        }
        __syncthreads();
        if (!abort_flag) {
            // (3) each miss's slot (a free one, else its victim; the victim's owner loses it),
            //     and the order of the appended slots: hits then misses, ascending id;
            int ms = -1;
            if (miss_t) {
                if (rm < n_free) {
                    ms = filled + rm;
                } else {
                    ms = vict[rm - n_free];
                    const int o = owner[ms];
                    if (o >= key0 && o < key0 + E) slot_l[o - key0] = -1;  // not requested: no other writer
                    else if (o >= 0 && o < n_keys) g_slot_of[o] = -1;
                }
                app[nh + rm] = ms;
            }
            if (hit_t) app[rh] = slot_l[e_t];
            const int old_tail = s_tail;
            const uint32_t ep_new = s_hd.epoch + 1u;  // read before thread 0 advances it below
            __syncthreads();
            // (4) append them at the tail
            const int na = nh + nm;
            for (int i = threadIdx.x; i < na; i += blockDim.x) {
                const int sa = app[i];
                prev[sa] = i == 0 ? old_tail : app[i - 1];
                next[sa] = i + 1 < na ? app[i + 1] : -1;
            }
            if (miss_t) {
                owner[ms] = key0 + e_t;
                slot_l[e_t] = ms;
                miss[e_t] = 1;
            }
            if (byp_t) miss[e_t] = 1;
            if (!speculative && (hit_t || miss_t)) g_recent[slot_l[e_t]] = ep_new;  // the slots of this request
            if (threadIdx.x == 0) {
                if (na > 0) {
                    if (old_tail >= 0) next[old_tail] = app[0];
                    else s_head = app[0];
                    s_tail = app[na - 1];
                }
                commit = 1;
                s_hd.head = s_head;
                s_hd.tail = s_tail;
                s_hd.n_filled = min(n_slots, filled + nm);
                if (speculative) {  // a prefetch: the same LRU rules, its own counters
                    s_hd.pf_queries += nh + nm + nbyp;
                    s_hd.pf_hits += nh;
                    s_hd.pf_fills += nm;
                    s_hd.evictions += m_evict;
                    s_hd.h2d_bytes += (uint64_t)nm * image_bytes;  // copied by the prefetch
                } else {
                    const int b = n_tokens <= 8 ? 0 : 1;
                    s_hd.queries[b] += nh + nm + nbyp;
                    s_hd.hits[b] += nh;
                    s_hd.misses[b] += nm + nbyp;
                    s_hd.evictions += m_evict;
                    s_hd.bypassed += nbyp;
                    s_hd.h2d_bytes += (uint64_t)(nm + nbyp) * image_bytes;  // read from host memory
                    s_hd.route_queries += n_real;
                    s_hd.ensure_calls += 1;
                    s_hd.epoch += 1;
                }
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && speculative && !commit && !abort_invalid) ((DevHeader *)state)->pf_aborts += 1;
    if (commit && !speculative) {  // routes whose expert was resident before this call (ids valid here)
        int h = 0;
        for (int i = threadIdx.x; i < n_ids; i += blockDim.x) h += s_ids[i] >= 0 && !miss[s_ids[i]];
        if (h) atomicAdd(&route_hits, h);
        __syncthreads();
        if (threadIdx.x == 0) s_hd.route_hits += route_hits;
    }
    __syncthreads();
    if (commit) {
        for (int i = threadIdx.x; i < (int)(sizeof(DevHeader) / 4); i += blockDim.x)
            ((int32_t *)hd)[i] = ((const int32_t *)&s_hd)[i];
        for (int i = threadIdx.x; i < n_slots; i += blockDim.x) {
            g_owner[i] = owner[i];
            g_prev[i] = prev[i];
            g_next[i] = next[i];
        }
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        if (commit) {
            g_slot_of[key0 + e] = slot_l[e];
            if (want[e] && !speculative) g_count[key0 + e] = cnt_l[e] + 1u;
        }
        table_out[e] = commit ? slot_l[e] : -1;
        src_out[e] = (commit && miss[e]) ? s_img[e] : 0ull;  // admitted misses and bypassed
    }
}

int dev_state_init(moe_cache *c) {
    const moe_cache_desc &d = c->d;
    const DevLayout L = dev_layout(d.n_layers, d.n_experts, d.n_slots);
    std::vector<uint8_t> h(L.total, 0);
    DevHeader *hd = (DevHeader *)h.data();
    hd->n_filled = 0;
    hd->head = -1;
    hd->tail = -1;
    const size_t nk = (size_t)d.n_layers * d.n_experts;
    int32_t *slot_of = (int32_t *)(h.data() + L.slot_of);
    for (size_t i = 0; i < nk; ++i) slot_of[i] = -1;
    int32_t *owner = (int32_t *)(h.data() + L.owner), *prev = (int32_t *)(h.data() + L.prev),
            *next = (int32_t *)(h.data() + L.next);
    for (int s = 0; s < d.n_slots; ++s) owner[s] = prev[s] = next[s] = -1;
    uint64_t *img = (uint64_t *)(h.data() + L.img);
    for (size_t i = 0; i < nk; ++i) img[i] = (uint64_t)(uintptr_t)c->images[i];
    MOE_TRY_CUDA(cudaMemcpy(d.device_state, h.data(), L.total, cudaMemcpyHostToDevice));
    return MOE_OK;
}

}  // namespace

extern "C" int moe_cache_state_bytes(int n_layers, int n_experts, int n_slots, size_t *bytes) {
    MOE_CHECK(bytes && n_layers >= 1 && n_experts >= 1 && n_experts <= MOE_MAX_E && n_slots >= 1);
    *bytes = dev_layout(n_layers, n_experts, n_slots).total;
    return MOE_OK;
}

static int plan_launch(moe_cache *c, int layer, const int32_t *d_ids, int n_tokens, int k, int32_t *d_table_out,
                       uint64_t *d_fill_src_out, moe_stream_t s, int speculative) {
    MOE_CHECK(c && c->d.device_managed && d_ids && d_table_out && d_fill_src_out);
    MOE_CHECK(n_tokens >= 1 && n_tokens <= MOE_DECODE_MAX_T && k >= 1 && k <= MOE_MAX_K);
    const moe_cache_desc &d = c->d;
    const int ll = layer - d.first_layer;
    MOE_CHECK(ll >= 0 && ll < d.n_layers);
    const DevLayout L = dev_layout(d.n_layers, d.n_experts, d.n_slots);
    // owner, prev, next (int32 per slot), the layer's slots (int32 per expert), want and miss
    // (a byte per expert), the hit marks (a byte per slot)
    auto plan_smem = [](int n_slots, int E) { return (size_t)n_slots * 13 + (size_t)E * 10; };
    const size_t smem = plan_smem(d.n_slots, d.n_experts);
    {
        // the attribute belongs to the kernel on one device: set once per device
        static std::mutex mu;
        static bool attr_set[64] = {false};
        int dev = -1;
        MOE_TRY_CUDA(cudaGetDevice(&dev));
        if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            MOE_TRY_CUDA(cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              (int)plan_smem(MOE_PLAN_MAX_SLOTS, MOE_MAX_E)));
            attr_set[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    moe_pdl_config(&cfg, attr, dim3(1), dim3(256), smem, moe_cuda_stream(s));
    MOE_TRY_CUDA(cudaLaunchKernelEx(&cfg, plan_kernel, (uint8_t *)d.device_state, L, ll, d.n_experts, d.n_slots,
                                    d_ids, n_tokens, k, c->image_bytes, std::max(1, d.admit_after), speculative,
                                    d_table_out, d_fill_src_out, moe_status_word_device_ptr()));
    MOE_TRY_CUDA(cudaGetLastError());
    return MOE_OK;
}

extern "C" int moe_cache_plan(moe_cache *c, int layer, const int32_t *d_ids, int n_tokens, int k,
                              int32_t *d_table_out, uint64_t *d_fill_src_out, moe_stream_t s) {
    return plan_launch(c, layer, d_ids, n_tokens, k, d_table_out, d_fill_src_out, s, 0);
}

extern "C" int moe_cache_prefetch_plan(moe_cache *c, int layer, const int32_t *d_ids, int n_tokens, int k,
                                       int32_t *d_table_out, uint64_t *d_fill_src_out, moe_stream_t s) {
    return plan_launch(c, layer, d_ids, n_tokens, k, d_table_out, d_fill_src_out, s, 1);
}

namespace {
// Copies each expert's pinned host image (src[e] != 0) into its slot (table[e] >= 0): the CTAs
// split the experts' images into 16-byte pieces, eight in flight per thread.
__global__ void __launch_bounds__(256) prefetch_fill_kernel(const int32_t *__restrict__ table,
                                                            const uint64_t *__restrict__ src, int E,
                                                            uint8_t *__restrict__ pool, size_t slot_bytes,
                                                            size_t image_bytes, int n_slots) {
    const size_t n16 = image_bytes / 16;
    for (int e = 0; e < E; ++e) {
        const uint64_t sp = src[e];
        const int sl = table[e];
        if (sp == 0ull || sl < 0 || sl >= n_slots) continue;
        const uint4 *from = (const uint4 *)(uintptr_t)sp;
        uint4 *to = (uint4 *)(pool + (size_t)sl * slot_bytes);
        const size_t stride = (size_t)gridDim.x * blockDim.x;
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += 8 * stride) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (i + u * stride < n16) v[u] = __ldcs(from + i + u * stride);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (i + u * stride < n16) __stcg(to + i + u * stride, v[u]);
        }
    }
}
}  // namespace

extern "C" int moe_cache_prefetch_fill(moe_cache *c, const int32_t *d_table, const uint64_t *d_fill_src,
                                       moe_stream_t s) {
    MOE_CHECK(c && c->d.device_managed && d_table && d_fill_src);
    MOE_CHECK((c->image_bytes % 16) == 0);
    prefetch_fill_kernel<<<64, 256, 0, moe_cuda_stream(s)>>>(d_table, d_fill_src, c->d.n_experts,
                                                            (uint8_t *)c->d.device_pool, c->d.slot_bytes,
                                                            c->image_bytes, c->d.n_slots);
    MOE_TRY_CUDA(cudaGetLastError());
    return MOE_OK;
}

int moe_write_ints(int32_t *const dst[3], const int n[3], const int32_t *const src[3], cudaStream_t s) {
    IntPayload pay;
    for (int a = 0; a < 3; ++a) {
        if (n[a] < 0 || n[a] > MOE_MAX_E) return MOE_ERR_INVALID;
        for (int i = 0; i < n[a]; ++i) pay.v[a][i] = src[a][i];
    }
    write_ints_kernel<<<1, MOE_MAX_E, 0, s>>>(dst[0], n[0], dst[1], n[1], dst[2], n[2], pay);
    MOE_TRY_CUDA(cudaGetLastError());
    return MOE_OK;
}

extern "C" int moe_cache_create(const moe_cache_desc *desc, moe_cache **out) {
    MOE_CHECK(desc && out);
    *out = nullptr;
    const moe_cache_desc &d = *desc;
    MOE_CHECK(d.qtype == MOE_Q8_0 || d.qtype == MOE_Q4_SM);
    MOE_CHECK(d.H > 0 && d.F > 0 && d.H % 32 == 0 && d.F % 32 == 0);
    MOE_CHECK(d.n_layers >= 1 && d.n_experts >= 1 && d.n_experts <= MOE_MAX_E && d.first_layer >= 0);
    MOE_CHECK(d.n_slots >= 1);
    MOE_CHECK(d.admit_after >= 0 && d.lru_window >= 0);
    if (d.device_managed && d.lru_window > 0) return MOE_ERR_UNSUPPORTED;
    const size_t img = moe_expert_image_bytes(d.qtype, d.H, d.F);
    MOE_CHECK(d.slot_bytes >= img && d.slot_bytes % 256 == 0);
    MOE_CHECK(d.device_pool && ((uintptr_t)d.device_pool % 256) == 0);
    MOE_CHECK(d.host_images);
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, d.device_pool) != cudaSuccess || attr.type != cudaMemoryTypeDevice)
        return MOE_ERR_INVALID;
    const size_t n_img = (size_t)d.n_layers * d.n_experts;
    for (size_t i = 0; i < n_img; ++i) {
        const void *p = d.host_images[i];
        if (!p) return MOE_ERR_INVALID;
        if (cudaPointerGetAttributes(&attr, p) != cudaSuccess || attr.type != cudaMemoryTypeHost)
            return MOE_ERR_INVALID;  // not pinned (page-locked) host memory
    }
    if (d.device_managed) {
        MOE_CHECK(d.n_slots <= MOE_PLAN_MAX_SLOTS);
        MOE_CHECK(d.device_state && ((uintptr_t)d.device_state % 256) == 0);
        MOE_CHECK(d.device_state_bytes >= dev_layout(d.n_layers, d.n_experts, d.n_slots).total);
        if (cudaPointerGetAttributes(&attr, d.device_state) != cudaSuccess || attr.type != cudaMemoryTypeDevice)
            return MOE_ERR_INVALID;
    }
    moe_cache *c = new moe_cache();
    c->d = d;
    c->image_bytes = img;
    c->images.assign(d.host_images, d.host_images + n_img);
    if (d.device_managed) {
        const int rc = dev_state_init(c);
        if (rc != MOE_OK) {
            delete c;
            return rc;
        }
    }
    c->slot_of.assign(n_img, -1);
    c->owner.assign(d.n_slots, -1);
    c->stamp.assign(d.n_slots, 0);
    c->last_use.assign(d.n_slots, -1);
    c->count.assign(n_img, 0u);
    c->last_tok.assign(d.n_slots, 0ull);
    for (int i = 0; i < MOE_EVENT_RING; ++i) {
        if (cudaEventCreateWithFlags(&c->ring[i], cudaEventDisableTiming) != cudaSuccess) {
            moe_cache_destroy(c);
            return MOE_ERR_CUDA;
        }
    }
    if (cudaEventCreateWithFlags(&c->upload_done, cudaEventDisableTiming) != cudaSuccess) {
        moe_cache_destroy(c);
        return MOE_ERR_CUDA;
    }
    reset_state(c);
    *out = c;
    return MOE_OK;
}

extern "C" int moe_cache_ensure(moe_cache *c, int layer, const int32_t *ids_host, int n_tokens, int k,
                                int32_t *slots_host_out, int *n_miss_out, uint8_t *miss_mask_host_out,
                                int32_t *d_slot_table, moe_stream_t s) {
    MOE_CHECK(c && ids_host && slots_host_out && n_miss_out);
    MOE_CHECK(!c->d.device_managed);
    MOE_CHECK(n_tokens >= 0 && n_tokens <= MOE_DECODE_MAX_T && k >= 1 && k <= MOE_MAX_K);
    const moe_cache_desc &d = c->d;
    const int E = d.n_experts;
    const int ll = layer - d.first_layer;
    MOE_CHECK(ll >= 0 && ll < d.n_layers);
    const int n_ids = n_tokens * k;
    bool want[MOE_MAX_E] = {false};
    for (int i = 0; i < n_ids; ++i) {
        const int e = ids_host[i];
        if (e == -1) continue;  // a route dropped by the load threshold
        MOE_CHECK(e >= 0 && e < E);
        want[e] = true;
    }
    int n_distinct = 0;
    for (int e = 0; e < E; ++e) n_distinct += want[e];

    const int64_t key0 = (int64_t)ll * E;
    // the window: the token clock advances at the group's first layer; slots unused for more
    // than lru_window tokens are freed before the request (their experts miss)
    const uint64_t tok = c->tok + (layer == d.first_layer ? (uint64_t)n_tokens : 0ull);
    std::vector<int> stale;
    if (d.lru_window > 0)
        for (int sl = 0; sl < d.n_slots; ++sl)
            if (c->owner[sl] >= 0 && tok - c->last_tok[sl] > (uint64_t)d.lru_window) stale.push_back(sl);
    auto is_stale = [&](int sl) { return std::binary_search(stale.begin(), stale.end(), sl); };
    // admission: a miss takes a slot once its accesses (this one included) reach admit_after
    const uint32_t theta = (uint32_t)std::max(1, d.admit_after);
    bool hit[MOE_MAX_E] = {false}, bypass[MOE_MAX_E] = {false};
    int n_need = 0, n_bypass = 0;
    for (int e = 0; e < E; ++e) {
        if (!want[e]) continue;
        const int sl = c->slot_of[key0 + e];
        hit[e] = sl >= 0 && !is_stale(sl);
        bypass[e] = !hit[e] && c->count[key0 + e] + 1 < theta;
        n_need += !bypass[e];
        n_bypass += bypass[e];
    }
    if (n_need > d.n_slots) return MOE_ERR_CAPACITY;  // nothing has changed
    if (miss_mask_host_out)  // 1 only for the experts this call uploads
        for (int e = 0; e < E; ++e) miss_mask_host_out[e] = 0;
    c->tok = tok;
    for (int sl : stale) {
        c->lru.erase({c->stamp[sl], sl});
        c->slot_of[c->owner[sl]] = -1;
        c->owner[sl] = -1;
        c->free_slots.insert(sl);
        c->st.window_evictions++;
    }
    for (int e = 0; e < E; ++e)
        if (want[e]) c->count[key0 + e]++;
    // 1. hits, ascending id: most recent
    for (int e = 0; e < E; ++e) {
        if (!hit[e]) continue;
        const int sl = c->slot_of[key0 + e];
        c->lru.erase({c->stamp[sl], sl});
        c->stamp[sl] = ++c->clock;
        c->lru.insert({c->stamp[sl], sl});
        c->last_tok[sl] = tok;
    }
    // 2. misses, ascending id: lowest free slot, else LRU slot outside this request
    cudaStream_t cs = moe_cuda_stream(d.copy_stream);
    int n_miss = 0;
    uint64_t bytes = 0;
    int waited[MOE_EVENT_RING];
    int n_waited = 0;
    for (int e = 0; e < E; ++e) {
        if (!want[e] || hit[e] || bypass[e]) continue;
        int sl;
        bool evicted = false;
        if (!c->free_slots.empty()) {
            sl = *c->free_slots.begin();
            c->free_slots.erase(c->free_slots.begin());
        } else {
            auto it = c->lru.begin();
            while (it != c->lru.end()) {
                const int64_t o = c->owner[it->second];
                if (!(o >= key0 && o < key0 + E && want[o - key0])) break;
                ++it;
            }
            if (it == c->lru.end()) return MOE_ERR_CAPACITY;  // unreachable when n_distinct <= n_slots
            sl = it->second;
            c->lru.erase(it);
            c->slot_of[c->owner[sl]] = -1;
            c->owner[sl] = -1;
            evicted = true;
        }
        // upload: wait for the slot's last reader, then copy the pinned image
        bool failed = moe_fault_take_upload();
        if (!failed && c->last_use[sl] >= 0) {
            const int ev = c->last_use[sl];
            bool seen = false;
            for (int i = 0; i < n_waited; ++i) seen |= waited[i] == ev;
            if (!seen) {
                failed = cudaStreamWaitEvent(cs, c->ring[ev], 0) != cudaSuccess;
                waited[n_waited++] = ev;
            }
        }
        if (!failed)
            failed = cudaMemcpyAsync((char *)d.device_pool + (size_t)sl * d.slot_bytes,
                                     c->images[key0 + e], c->image_bytes, cudaMemcpyHostToDevice,
                                     cs) != cudaSuccess;
        if (failed) {
            // the slot stays empty; the pool is consistent; this call's stats are not counted
            c->last_use[sl] = -1;
            c->free_slots.insert(sl);
            if (n_miss > 0 && cudaEventRecord(c->upload_done, cs) == cudaSuccess) c->upload_pending = true;
            return MOE_ERR_CUDA;
        }
        c->owner[sl] = key0 + e;
        c->slot_of[key0 + e] = sl;
        c->stamp[sl] = ++c->clock;
        c->lru.insert({c->stamp[sl], sl});
        c->last_tok[sl] = tok;
        c->last_use[sl] = -1;
        if (evicted) c->st.evictions++;
        ++n_miss;
        bytes += c->image_bytes;
        if (miss_mask_host_out) miss_mask_host_out[e] = 1;
    }
    if (n_miss > 0) {
        MOE_TRY_CUDA(cudaEventRecord(c->upload_done, cs));
        c->upload_pending = true;
    } else {
        c->upload_pending = false;
    }

    c->last_slots.clear();
    for (int e = 0; e < E; ++e)
        if (want[e] && !bypass[e]) c->last_slots.push_back(c->slot_of[key0 + e]);
    int route_hits = 0, n_real = 0;
    for (int i = 0; i < n_ids; ++i) {
        const int e = ids_host[i];
        slots_host_out[i] = e < 0 ? -1 : c->slot_of[key0 + e];
        route_hits += e >= 0 && hit[e];
        n_real += e >= 0;
    }
    *n_miss_out = n_miss;
    const int bucket = n_tokens <= 8 ? 0 : 1;
    c->st.queries[bucket] += n_distinct;
    c->st.hits[bucket] += n_distinct - n_miss - n_bypass;
    c->st.misses[bucket] += n_miss + n_bypass;
    c->st.bypassed += n_bypass;
    c->st.h2d_bytes += bytes + (uint64_t)n_bypass * c->image_bytes;  // read from host memory
    c->st.route_queries += n_real;
    c->st.route_hits += route_hits;
    c->st.ensure_calls++;

    if (d_slot_table) {
        int32_t *dst[3] = {d_slot_table, nullptr, nullptr};
        const int n[3] = {E, 0, 0};
        const int32_t *src[3] = {&c->slot_of[key0], nullptr, nullptr};
        const int rc = moe_write_ints(dst, n, src, moe_cuda_stream(s));
        if (rc != MOE_OK) return rc;
    }
    return MOE_OK;
}

extern "C" int moe_cache_wait_uploads(moe_cache *c, moe_stream_t s) {
    MOE_CHECK(c && !c->d.device_managed);
    if (c->upload_pending) MOE_TRY_CUDA(cudaStreamWaitEvent(moe_cuda_stream(s), c->upload_done, 0));
    return MOE_OK;
}

extern "C" int moe_cache_release(moe_cache *c, moe_stream_t s) {
    MOE_CHECK(c && !c->d.device_managed);
    if (c->last_slots.empty()) return MOE_OK;
    const int ev = c->ring_next;
    MOE_TRY_CUDA(cudaEventRecord(c->ring[ev], moe_cuda_stream(s)));
    c->ring_next = (c->ring_next + 1) % MOE_EVENT_RING;
    for (int sl : c->last_slots) c->last_use[sl] = ev;
    c->last_slots.clear();
    return MOE_OK;
}

extern "C" int moe_cache_stats_get(const moe_cache *c, moe_cache_stats *out) {
    MOE_CHECK(c && out);
    if (c->d.device_managed) {
        DevHeader h;
        MOE_TRY_CUDA(cudaDeviceSynchronize());
        MOE_TRY_CUDA(cudaMemcpy(&h, c->d.device_state, sizeof h, cudaMemcpyDeviceToHost));
        moe_cache_stats st{};
        for (int b = 0; b < 2; ++b) {
            st.queries[b] = h.queries[b];
            st.hits[b] = h.hits[b];
            st.misses[b] = h.misses[b];
        }
        st.evictions = h.evictions;
        st.h2d_bytes = h.h2d_bytes;
        st.route_queries = h.route_queries;
        st.route_hits = h.route_hits;
        st.ensure_calls = h.ensure_calls;
        st.bypassed = h.bypassed;
        st.window_evictions = h.window_evictions;
        st.prefetch_queries = h.pf_queries;
        st.prefetch_hits = h.pf_hits;
        st.prefetch_fills = h.pf_fills;
        st.prefetch_aborts = h.pf_aborts;
        *out = st;
        return MOE_OK;
    }
    *out = c->st;
    return MOE_OK;
}

extern "C" int moe_cache_reset(moe_cache *c) {
    MOE_CHECK(c);
    if (c->d.device_managed) {
        MOE_TRY_CUDA(cudaDeviceSynchronize());
        return dev_state_init(c);
    }
    // wait for in-flight uploads and readers so that no copy lands in a slot reused later
    MOE_TRY_CUDA(cudaStreamSynchronize(moe_cuda_stream(c->d.copy_stream)));
    for (int i = 0; i < MOE_EVENT_RING; ++i) MOE_TRY_CUDA(cudaEventSynchronize(c->ring[i]));
    reset_state(c);
    return MOE_OK;
}

extern "C" void moe_cache_destroy(moe_cache *c) {
    if (!c) return;
    if (c->d.copy_stream) cudaStreamSynchronize(moe_cuda_stream(c->d.copy_stream));
    for (int i = 0; i < MOE_EVENT_RING; ++i)
        if (c->ring[i]) cudaEventDestroy(c->ring[i]);
    if (c->upload_done) cudaEventDestroy(c->upload_done);
    delete c;
}

const void *moe_cache_image(const moe_cache *c, int layer, int expert) {
    if (!c) return nullptr;
    const int ll = layer - c->d.first_layer;
    if (ll < 0 || ll >= c->d.n_layers || expert < 0 || expert >= c->d.n_experts) return nullptr;
    return c->images[(size_t)ll * c->d.n_experts + expert];
}

extern "C" int moe_cache_lookup(const moe_cache *c, int layer, int expert) {
    if (!c) return -1;
    const int ll = layer - c->d.first_layer;
    if (ll < 0 || ll >= c->d.n_layers || expert < 0 || expert >= c->d.n_experts) return -1;
    if (c->d.device_managed) {
        const DevLayout L = dev_layout(c->d.n_layers, c->d.n_experts, c->d.n_slots);
        int32_t v = -1;
        if (cudaDeviceSynchronize() != cudaSuccess) return -1;
        if (cudaMemcpy(&v, (const uint8_t *)c->d.device_state + L.slot_of +
                               ((size_t)ll * c->d.n_experts + expert) * 4,
                       4, cudaMemcpyDeviceToHost) != cudaSuccess)
            return -1;
        return v;
    }
    return c->slot_of[(size_t)ll * c->d.n_experts + expert];
}

extern "C" int moe_slots_for_budget(size_t budget_bytes, const size_t *per_expert_bytes, int n_groups,
                                    int k, int *slots_out) {
    MOE_CHECK(per_expert_bytes && slots_out && n_groups >= 1 && k >= 1);
    size_t sum = 0;
    for (int g = 0; g < n_groups; ++g) {
        MOE_CHECK(per_expert_bytes[g] > 0);
        sum += per_expert_bytes[g];
    }
    const size_t n = budget_bytes / sum;
    if (n < (size_t)k + 1) {
        for (int g = 0; g < n_groups; ++g) slots_out[g] = 0;
        return MOE_ERR_BUDGET;
    }
    for (int g = 0; g < n_groups; ++g) slots_out[g] = (int)(n > 0x7FFFFFFF ? 0x7FFFFFFF : n);
    return MOE_OK;
}

const void *moe_cache_pool(const moe_cache *c, int *n_slots) {
    if (n_slots) *n_slots = c ? c->d.n_slots : 0;
    return c ? c->d.device_pool : nullptr;
}

bool moe_cache_is_device_managed(const moe_cache *c) { return c && c->d.device_managed; }

int moe_cache_layer_range(const moe_cache *c, int *first_layer, int *n_layers) {
    MOE_CHECK(c && first_layer && n_layers);
    *first_layer = c->d.first_layer;
    *n_layers = c->d.n_layers;
    return MOE_OK;
}
