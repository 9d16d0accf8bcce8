// moe_expert_ffn_noalloc — the expert FFN with its scratch memory inside the library.
//
// moe_expert_ffn needs a scratch workspace (route lists and the gate/up partial sums)
// that the caller allocates.  Some callers cannot allocate device memory at all: a
// plugin running inside a host framework that owns every device allocation and hands
// the plugin only its input and output tensors, or a latency-critical decode loop in
// which a cudaMalloc/cudaFree (which may synchronise the whole device) is not allowed.
// This entry point serves them: its scratch is one statically sized array in device
// memory that exists on every device where the library is loaded, for the life of the
// process.  It runs exactly the same kernels as moe_expert_ffn.
#include <mutex>

#include "moe_common.cuh"

// Size of the library-owned scratch array (per device): MOE_NOALLOC_SCRATCH_MAX (moe.h).
#define MOE_NOALLOC_SCRATCH_BYTES MOE_NOALLOC_SCRATCH_MAX

static __device__ __align__(256) unsigned char g_moe_ffn_scratch[MOE_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the scratch array for the current device.  The host-side symbol
// is only a stand-in, so the address is resolved once per device (with that device
// current) and cached.
int noalloc_scratch(void **out) {
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    int dev = -1;
    MOE_TRY_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_moe_ffn_scratch);
        if (e != cudaSuccess) {
            moe_note_cuda_error(e);   // reported by moe_last_cuda_error
            (void)cudaGetLastError(); // not left behind for the next caller
            return MOE_ERR_CUDA;
        }
        if (!p) return MOE_ERR_CUDA;
        addr[dev] = p;
    }
    *out = addr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" int moe_expert_ffn_noalloc(const void *x, int xtype, int T, int H, int F, int qtype, int E,
                                      int k, const int32_t *ids, const float *weights,
                                      const int32_t *d_slot_table, int n_slots, const void *pool,
                                      size_t slot_bytes, const int32_t *expert_subset, int n_subset,
                                      float *partial, moe_stream_t s) {
    MOE_CHECK(T >= 0 && H > 0 && F > 0 && H % 32 == 0 && F % 32 == 0);
    MOE_CHECK(qtype == MOE_Q8_0 || qtype == MOE_Q4_SM);
    MOE_CHECK(E >= 1 && E <= MOE_MAX_E && k >= 1 && k <= MOE_MAX_K && k <= E);
    MOE_CHECK(xtype == MOE_F32 || xtype == MOE_BF16);
    if (moe_ffn_workspace_bytes(T, H, F, qtype, xtype, E, k) > MOE_NOALLOC_SCRATCH_BYTES)
        return MOE_ERR_UNSUPPORTED;  // the request needs more scratch than the static array holds
    void *scratch = nullptr;
    const int rc = noalloc_scratch(&scratch);
    if (rc != MOE_OK) return rc;
    // Every scratch word the kernels read is written earlier in the same call, so the
    // array needs no clearing between calls.
    return moe_expert_ffn_impl(x, xtype, T, H, F, qtype, E, k, ids, weights, d_slot_table, n_slots,
                               pool, slot_bytes, expert_subset, n_subset, partial, scratch,
                               MOE_NOALLOC_SCRATCH_BYTES, moe_cuda_stream(s), nullptr);
}
