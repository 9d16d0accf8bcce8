// Status strings, the per-device status word and host-side fault injection.
#include <atomic>
#include <mutex>

#include "moe_common.cuh"

// One word per device (a __device__ variable exists once per device context).
static __device__ int g_moe_status_word;

extern "C" const char *moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID: return "invalid argument";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_CAPACITY: return "more distinct experts requested than the pool has slots";
        case MOE_ERR_BUDGET: return "budget too small for one request in every group";
        case MOE_ERR_TIMEOUT: return "a bounded device-side wait ran out";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape or type";
        default: return "unknown status";
    }
}

static thread_local cudaError_t g_last_cuda_error = cudaSuccess;

void moe_note_cuda_error(cudaError_t e) { g_last_cuda_error = e; }

extern "C" const char *moe_last_cuda_error(void) {
    return g_last_cuda_error == cudaSuccess ? "none" : cudaGetErrorName(g_last_cuda_error);
}

int *moe_status_word_device_ptr() {
    static std::mutex mu;
    static int *ptrs[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_moe_status_word) != cudaSuccess) return nullptr;
        ptrs[dev] = (int *)p;
    }
    return ptrs[dev];
}

extern "C" int moe_device_status(int *status_out, int clear) {
    MOE_CHECK(status_out);
    int v = 0;
    MOE_TRY_CUDA(cudaDeviceSynchronize());
    MOE_TRY_CUDA(cudaMemcpyFromSymbol(&v, g_moe_status_word, sizeof(int)));
    if (clear) {
        int z = 0;
        MOE_TRY_CUDA(cudaMemcpyToSymbol(g_moe_status_word, &z, sizeof(int)));
    }
    *status_out = v;
    return MOE_OK;
}

// ------------------------------------------------------------------ fault injection

static std::atomic<int> g_fault_kind{0};
static std::atomic<int> g_fault_countdown{0};

extern "C" int moe_debug_inject_fault(int kind, int countdown) {
    MOE_CHECK(kind == 0 || kind == 1 || kind == 2);
    MOE_CHECK(countdown >= 0);
    g_fault_countdown.store(countdown);
    g_fault_kind.store(kind);
    return MOE_OK;
}

bool moe_fault_take_grid_barrier() {
    if (g_fault_kind.load() != 2) return false;
    int c = g_fault_countdown.fetch_sub(1);
    if (c == 0) {
        g_fault_kind.store(0);
        return true;
    }
    return false;
}

bool moe_fault_take_upload() {
    if (g_fault_kind.load() != 1) return false;
    int c = g_fault_countdown.fetch_sub(1);
    if (c == 0) {
        g_fault_kind.store(0);
        return true;
    }
    return false;
}
