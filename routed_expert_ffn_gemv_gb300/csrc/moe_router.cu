// Router GEMV + top-k + softmax over the selected experts (R1).
//
// Gating as on page 1 ("llama.cpp MoE 模型卸载", section 3.1): logits = x.W_r + b,
// then the k largest, then a softmax — here taken over the k selected logits, which
// equals a full softmax renormalised over the selected experts; equal logits are
// ordered by ascending expert id.  Page 1 also batches the gating of several tokens
// into one matrix product (section 5.2); one launch here handles every token.
//
// GB300 mapping: a cluster of MOE_ROUTER_CLUSTER CTAs per group of up to 32 tokens.
// CTA r of the cluster owns rows [r*H/C, (r+1)*H/C) of W_r [H][E]: one bulk copy
// (TMA engine) brings that contiguous slice into shared memory, the CTA computes
// partial logits for its rows, and cluster rank 0 sums the C partials over
// distributed shared memory in rank order, adds the bias and selects the top-k
// with one warp per token.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "moe_ptx.cuh"

#define MOE_ROUTER_CLUSTER 8
#define MOE_ROUTER_TOKENS 32   // tokens per cluster
#define MOE_ROUTER_CHUNK 8     // tokens accumulated at once in registers
#define MOE_ROUTER_THREADS 256

namespace {

struct RouterSmem {
    // offsets (bytes) into dynamic shared memory
    size_t w, x, red, part, bar, total;
};

__host__ __device__ inline RouterSmem router_smem_layout(int H, int E) {
    RouterSmem L;
    const int HS = H / MOE_ROUTER_CLUSTER;
    const int NP = (E + 1) / 2;
    const int HSUB = MOE_ROUTER_THREADS / NP;
    size_t off = 0;
    L.w = off;     off += ((size_t)HS * E * 2 + 15) / 16 * 16 + 16;   // + pad for the odd-E pair
    L.x = off;     off += (size_t)MOE_ROUTER_TOKENS * HS * 4;
    L.red = off;   off += (size_t)HSUB * MOE_ROUTER_CHUNK * NP * 2 * 4;
    L.part = off;  off += (size_t)MOE_ROUTER_TOKENS * E * 4;
    L.bar = off;   off += 16;
    L.total = off;
    return L;
}

template <int XT>
__device__ __forceinline__ float load_x(const void *x, size_t i) {
    if (XT == MOE_BF16) return __bfloat162float(((const __nv_bfloat16 *)x)[i]);
    return ((const float *)x)[i];
}

// (v, id) ordering of the selection: larger logit first, then lower id.
__device__ __forceinline__ bool better(float v1, int i1, float v2, int i2) {
    return v1 > v2 || (v1 == v2 && i1 < i2);
}

template <int XT>
__global__ void __launch_bounds__(MOE_ROUTER_THREADS)
router_topk_kernel(const void *__restrict__ x, int T, int H, const uint16_t *__restrict__ w_router,
                   const float *__restrict__ bias, int E, int k, int32_t *__restrict__ ids,
                   float *__restrict__ weights, float *__restrict__ logits_out, int use_bulk,
                   int *status) {
    extern __shared__ __align__(128) unsigned char smem[];
    const RouterSmem L = router_smem_layout(H, E);
    const uint16_t *w_s = (const uint16_t *)(smem + L.w);
    float *x_s = (float *)(smem + L.x);
    float *red = (float *)(smem + L.red);
    float *part = (float *)(smem + L.part);
    uint64_t *bar = (uint64_t *)(smem + L.bar);

    const int rank = (int)cluster_ctarank();
    const int HS = H / MOE_ROUTER_CLUSTER;
    const int h0 = rank * HS;
    const int t0 = blockIdx.y * MOE_ROUTER_TOKENS;
    const int TT = min(MOE_ROUTER_TOKENS, T - t0);
    const int tid = threadIdx.x;
    const size_t wbytes = (size_t)HS * E * 2;

    // ---- W_r slice -> shared memory (bulk copy when aligned, else plain loads)
    bool w_ok = true;
    if (use_bulk) {
        if (tid == 0) {
            mbar_init(bar, 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(bar, (uint32_t)wbytes);
            bulk_g2s((void *)w_s, w_router + (size_t)h0 * E, (uint32_t)wbytes, bar);
        }
    } else {
        for (size_t i = tid; i < (size_t)HS * E; i += MOE_ROUTER_THREADS)
            ((uint16_t *)w_s)[i] = w_router[(size_t)h0 * E + i];
    }
    if (tid == 0) ((uint16_t *)w_s)[(size_t)HS * E] = 0;  // pad read by the odd-E pair
    // ---- x slice of this cluster's tokens
    for (int i = tid; i < TT * HS; i += MOE_ROUTER_THREADS) {
        const int t = i / HS, h = i % HS;
        x_s[i] = load_x<XT>(x, (size_t)(t0 + t) * H + h0 + h);
    }
    __syncthreads();
    if (use_bulk) w_ok = mbar_wait_bounded(bar, 0, status);

    const int NP = (E + 1) / 2;
    const int HSUB = MOE_ROUTER_THREADS / NP;
    const int pair = tid % NP, hsub = tid / NP;
    const bool active = hsub < HSUB;

    for (int c0 = 0; c0 < TT; c0 += MOE_ROUTER_CHUNK) {
        float acc0[MOE_ROUTER_CHUNK], acc1[MOE_ROUTER_CHUNK];
#pragma unroll
        for (int t = 0; t < MOE_ROUTER_CHUNK; ++t) acc0[t] = acc1[t] = 0.f;
        const int nt = min(MOE_ROUTER_CHUNK, TT - c0);
        if (active && w_ok) {
            for (int h = hsub; h < HS; h += HSUB) {
                // column 2*pair+1 == E (odd E) reads the next row or the pad; it is never stored
                const float w0 = __half2float(__ushort_as_half(w_s[(size_t)h * E + 2 * pair]));
                const float w1 = __half2float(__ushort_as_half(w_s[(size_t)h * E + 2 * pair + 1]));
#pragma unroll
                for (int t = 0; t < MOE_ROUTER_CHUNK; ++t) {
                    if (t < nt) {
                        const float xv = x_s[(c0 + t) * HS + h];
                        acc0[t] = fmaf(xv, w0, acc0[t]);
                        acc1[t] = fmaf(xv, w1, acc1[t]);
                    }
                }
            }
        }
        if (active) {
#pragma unroll
            for (int t = 0; t < MOE_ROUTER_CHUNK; ++t) {
                red[((size_t)hsub * MOE_ROUTER_CHUNK + t) * NP * 2 + 2 * pair] = acc0[t];
                red[((size_t)hsub * MOE_ROUTER_CHUNK + t) * NP * 2 + 2 * pair + 1] = acc1[t];
            }
        }
        __syncthreads();
        for (int i = tid; i < nt * E; i += MOE_ROUTER_THREADS) {
            const int t = i / E, e = i % E;
            float s = 0.f;
            for (int hs = 0; hs < HSUB; ++hs) s += red[((size_t)hs * MOE_ROUTER_CHUNK + t) * NP * 2 + e];
            part[(size_t)(c0 + t) * E + e] = s;
        }
        __syncthreads();
    }

    cluster_sync_all();  // every CTA's partial logits are complete and visible

    if (rank == 0) {
        const int warp = tid / 32, lane = tid % 32;
        constexpr int NPL = MOE_MAX_E / 32;
        for (int t = warp; t < TT; t += MOE_ROUTER_THREADS / 32) {
            float v[NPL];
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                const int e = lane + 32 * i;
                v[i] = -INFINITY;
                if (e < E) {
                    float s = 0.f;
                    for (int r = 0; r < MOE_ROUTER_CLUSTER; ++r)
                        s += ld_cluster_f32(cluster_map(&part[(size_t)t * E + e], r));
                    if (bias) s += bias[e];
                    if (logits_out) logits_out[(size_t)(t0 + t) * E + e] = s;
                    v[i] = (s != s) ? -INFINITY : s;  // NaN never wins
                }
            }
            unsigned taken = 0;
            float sel_v[MOE_MAX_K];
            int sel_i[MOE_MAX_K];
            for (int j = 0; j < k; ++j) {
                float bv = -INFINITY;
                int bi = 0x7FFFFFFF;
#pragma unroll
                for (int i = 0; i < NPL; ++i) {
                    const int e = lane + 32 * i;
                    if (e < E && !(taken >> i & 1u) && better(v[i], e, bv, bi)) {
                        bv = v[i];
                        bi = e;
                    }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                    if (better(ov, oi, bv, bi)) {
                        bv = ov;
                        bi = oi;
                    }
                }
                if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
                sel_v[j] = bv;
                sel_i[j] = bi;
            }
            float denom = 0.f;
            for (int j = 0; j < k; ++j) denom += expf(sel_v[j] - sel_v[0]);
            if (lane < k) {
                float myv = sel_v[0];
                int myi = sel_i[0];
                for (int j = 1; j < k; ++j)
                    if (j == lane) {
                        myv = sel_v[j];
                        myi = sel_i[j];
                    }
                ids[(size_t)(t0 + t) * k + lane] = myi;
                weights[(size_t)(t0 + t) * k + lane] = expf(myv - sel_v[0]) / denom;
            }
        }
    }
    cluster_sync_all();  // rank 0 has finished reading the other CTAs' shared memory
}

}  // namespace

extern "C" int moe_router_topk(const void *x, int xtype, int T, int H, const uint16_t *w_router,
                               const float *bias, int E, int k, int32_t *ids, float *weights,
                               float *logits, moe_stream_t s) {
    MOE_CHECK(T >= 0);
    MOE_CHECK(xtype == MOE_F32 || xtype == MOE_BF16);
    MOE_CHECK(H > 0 && H % 32 == 0);
    MOE_CHECK(E >= 1 && E <= MOE_MAX_E && k >= 1 && k <= MOE_MAX_K && k <= E);
    if (T == 0) return MOE_OK;
    MOE_CHECK(x && w_router && ids && weights);
    const RouterSmem L = router_smem_layout(H, E);
    if (L.total > 200 * 1024) return MOE_ERR_UNSUPPORTED;
    const int HS = H / MOE_ROUTER_CLUSTER;
    const size_t wbytes = (size_t)HS * E * 2;
    const int use_bulk = ((uintptr_t)w_router % 16 == 0) && (wbytes % 16 == 0) &&
                         (((size_t)HS * E * 2) % 16 == 0);
    int *status = moe_status_word_device_ptr();

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(MOE_ROUTER_CLUSTER, (T + MOE_ROUTER_TOKENS - 1) / MOE_ROUTER_TOKENS, 1);
    cfg.blockDim = dim3(MOE_ROUTER_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = moe_cuda_stream(s);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = MOE_ROUTER_CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (xtype == MOE_F32) {
        MOE_TRY_CUDA(cudaFuncSetAttribute(router_topk_kernel<MOE_F32>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total));
        MOE_TRY_CUDA(cudaLaunchKernelEx(&cfg, router_topk_kernel<MOE_F32>, x, T, H, w_router, bias, E,
                                        k, ids, weights, logits, use_bulk, status));
    } else {
        MOE_TRY_CUDA(cudaFuncSetAttribute(router_topk_kernel<MOE_BF16>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total));
        MOE_TRY_CUDA(cudaLaunchKernelEx(&cfg, router_topk_kernel<MOE_BF16>, x, T, H, w_router, bias,
                                        E, k, ids, weights, logits, use_bulk, status));
    }
    return MOE_OK;
}
