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
#include <set>
#include <utility>
#include <vector>

#include "moe_common.cuh"

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
}

}  // namespace

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
    moe_cache *c = new moe_cache();
    c->d = d;
    c->image_bytes = img;
    c->images.assign(d.host_images, d.host_images + n_img);
    c->slot_of.assign(n_img, -1);
    c->owner.assign(d.n_slots, -1);
    c->stamp.assign(d.n_slots, 0);
    c->last_use.assign(d.n_slots, -1);
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
    MOE_CHECK(n_tokens >= 0 && n_tokens <= MOE_DECODE_MAX_T && k >= 1 && k <= MOE_MAX_K);
    const moe_cache_desc &d = c->d;
    const int E = d.n_experts;
    const int ll = layer - d.first_layer;
    MOE_CHECK(ll >= 0 && ll < d.n_layers);
    const int n_ids = n_tokens * k;
    bool want[MOE_MAX_E] = {false};
    for (int i = 0; i < n_ids; ++i) {
        const int e = ids_host[i];
        MOE_CHECK(e >= 0 && e < E);
        want[e] = true;
    }
    int n_distinct = 0;
    for (int e = 0; e < E; ++e) n_distinct += want[e];
    if (n_distinct > d.n_slots) return MOE_ERR_CAPACITY;

    const int64_t key0 = (int64_t)ll * E;
    bool hit[MOE_MAX_E] = {false};
    // 1. hits, ascending id: most recent
    for (int e = 0; e < E; ++e) {
        if (!want[e]) continue;
        const int sl = c->slot_of[key0 + e];
        if (sl < 0) continue;
        hit[e] = true;
        c->lru.erase({c->stamp[sl], sl});
        c->stamp[sl] = ++c->clock;
        c->lru.insert({c->stamp[sl], sl});
    }
    // 2. misses, ascending id: lowest free slot, else LRU slot outside this request
    cudaStream_t cs = moe_cuda_stream(d.copy_stream);
    int n_miss = 0;
    uint64_t bytes = 0;
    int waited[MOE_EVENT_RING];
    int n_waited = 0;
    for (int e = 0; e < E; ++e) {
        if (!want[e] || hit[e]) continue;
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
    if (miss_mask_host_out)
        for (int e = 0; e < E; ++e)
            if (!(want[e] && !hit[e])) miss_mask_host_out[e] = 0;

    c->last_slots.clear();
    for (int e = 0; e < E; ++e)
        if (want[e]) c->last_slots.push_back(c->slot_of[key0 + e]);
    int route_hits = 0;
    for (int i = 0; i < n_ids; ++i) {
        slots_host_out[i] = c->slot_of[key0 + ids_host[i]];
        route_hits += hit[ids_host[i]];
    }
    *n_miss_out = n_miss;
    const int bucket = n_tokens <= 8 ? 0 : 1;
    c->st.queries[bucket] += n_distinct;
    c->st.hits[bucket] += n_distinct - n_miss;
    c->st.misses[bucket] += n_miss;
    c->st.h2d_bytes += bytes;
    c->st.route_queries += n_ids;
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
    MOE_CHECK(c);
    if (c->upload_pending) MOE_TRY_CUDA(cudaStreamWaitEvent(moe_cuda_stream(s), c->upload_done, 0));
    return MOE_OK;
}

extern "C" int moe_cache_release(moe_cache *c, moe_stream_t s) {
    MOE_CHECK(c);
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
    *out = c->st;
    return MOE_OK;
}

extern "C" int moe_cache_reset(moe_cache *c) {
    MOE_CHECK(c);
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

extern "C" int moe_cache_lookup(const moe_cache *c, int layer, int expert) {
    if (!c) return -1;
    const int ll = layer - c->d.first_layer;
    if (ll < 0 || ll >= c->d.n_layers || expert < 0 || expert >= c->d.n_experts) return -1;
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

int moe_cache_layer_range(const moe_cache *c, int *first_layer, int *n_layers) {
    MOE_CHECK(c && first_layer && n_layers);
    *first_layer = c->d.first_layer;
    *n_layers = c->d.n_layers;
    return MOE_OK;
}
