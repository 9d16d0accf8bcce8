// Internal helpers shared by libmoe's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

// Records the CUDA error behind an MOE_ERR_CUDA (see moe_last_cuda_error).
void moe_note_cuda_error(cudaError_t e);

#define MOE_TRY_CUDA(expr)                                   \
    do {                                                     \
        cudaError_t moe_err__ = (expr);                      \
        if (moe_err__ != cudaSuccess) {                      \
            moe_note_cuda_error(moe_err__);                  \
            return MOE_ERR_CUDA;                             \
        }                                                    \
    } while (0)

#define MOE_CHECK(cond)                                      \
    do {                                                     \
        if (!(cond)) return MOE_ERR_INVALID;                 \
    } while (0)

static inline cudaStream_t moe_cuda_stream(moe_stream_t s) { return (cudaStream_t)s; }

// ------------------------------------------------------------------ slot image layout
//
// A matrix of R rows (output features) by K columns (reduction) is stored in 32-row tiles
// (one row per lane of a warp), each tile a run of "tile blocks", one per 32-column block
// along K, so that any K range of a tile is one contiguous run of bytes.  A tile block is
//   codes:  PPB pieces of 512 bytes (q8_0: 2, 4-bit: 1); piece p holds, for lane 0..31,
//           16 bytes of codes: q8_0 columns 16p .. 16p+15 of the block, one byte each, stored
//           as q + 128 (offset binary); 4-bit the block's 16 code bytes in canonical order.
//           Lane l's 16 bytes sit at 512 p + 16 ((l + 4 p) mod 32): the second q8_0 piece is
//           rotated by four rows, so that the decode GEMV's 8-byte loads of rows r..r+3 from
//           both pieces (one half-warp) fall on opposite halves of the shared-memory banks;
//   scales: 32 entries, fp16 d (q8_0) or fp16 d, fp16 m (4-bit), the entry of row (lane) l
//           at position moe_scale_pos(l) = 4 (l % 8) + l / 8, so that rows l, l+8, l+16,
//           l+24 are adjacent.
// An expert image is gate [F][H], up [F][H], down [H][F].

#define MOE_TILE_ROWS 32

__host__ __device__ static inline int moe_piece_cols(int qtype) { return qtype == MOE_Q8_0 ? 16 : 32; }
__host__ __device__ static inline int moe_pieces_per_block(int qtype) { return qtype == MOE_Q8_0 ? 2 : 1; }
__host__ __device__ static inline int moe_scale_entry_bytes(int qtype) { return qtype == MOE_Q8_0 ? 2 : 4; }
__host__ __device__ static inline int moe_block_bytes(int qtype) { return qtype == MOE_Q8_0 ? 34 : 20; }
// bytes of one tile block: 32 rows of one 32-column block, codes then scales
__host__ __device__ static inline int moe_tile_block_bytes(int qtype) {
    return MOE_TILE_ROWS * (qtype == MOE_Q8_0 ? 32 : 16) + MOE_TILE_ROWS * moe_scale_entry_bytes(qtype);
}
__host__ __device__ static inline int moe_scale_pos(int lane) { return 4 * (lane & 7) + (lane >> 3); }

__host__ __device__ static inline size_t moe_quant_bytes(int qtype, int R, int K) {
    return qtype == MOE_Q8_0 ? (size_t)R * K : (size_t)R * K / 2;
}
__host__ __device__ static inline size_t moe_scale_bytes(int qtype, int R, int K) {
    return (size_t)R * (K / 32) * moe_scale_entry_bytes(qtype);
}
__host__ __device__ static inline size_t moe_matrix_bytes(int qtype, int R, int K) {
    return moe_quant_bytes(qtype, R, K) + moe_scale_bytes(qtype, R, K);
}
// byte offset of tile block (row tile g, block b) in a matrix
__host__ __device__ static inline size_t moe_tile_block_offset(int qtype, int K, int g, int b) {
    return ((size_t)g * (K / 32) + b) * moe_tile_block_bytes(qtype);
}
// within a tile block: the code bytes of lane l in piece p, and the scale entry of lane l
__host__ __device__ static inline int moe_piece_in_block(int p, int lane) { return p * 512 + ((lane + 4 * p) & 31) * 16; }
__host__ __device__ static inline int moe_scale_in_block(int qtype, int lane) {
    return MOE_TILE_ROWS * (qtype == MOE_Q8_0 ? 32 : 16) + moe_scale_pos(lane) * moe_scale_entry_bytes(qtype);
}
__host__ __device__ static inline size_t moe_expert_image_bytes(int qtype, int H, int F) {
    return 2 * moe_matrix_bytes(qtype, F, H) + moe_matrix_bytes(qtype, H, F);
}
// matrix m of an expert image: 0 gate, 1 up, 2 down
__host__ __device__ static inline size_t moe_expert_matrix_offset(int qtype, int H, int F, int m) {
    return (size_t)m * moe_matrix_bytes(qtype, F, H);
}

// ------------------------------------------------------------------ device status word

// Address of the current device's status word (see moe_device_status).
int *moe_status_word_device_ptr();

#define MOE_DEV_STATUS_OK 0

#ifdef __CUDACC__
__device__ static inline void moe_set_status(int *status_word, int code) {
    if (status_word) atomicCAS(status_word, 0, code);
}
#endif

// Host-side fault injection (tests): returns true if this miss upload must fail.
bool moe_fault_take_upload();
// Host-side fault injection (tests): returns true if this fused decode GEMV launch must be
// given a grid barrier that waits for an arrival that never comes (bounded, short).
bool moe_fault_take_grid_barrier();

// ------------------------------------------------------------------ decode FFN internals

struct moe_ffn_timing {
    // optional event pairs recorded around the kernels of one moe_expert_ffn call
    // (a null event is not recorded)
    cudaEvent_t permute0, permute1, gateup0, gateup1, down0, down1;
};

int moe_expert_ffn_impl(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k,
                        const int32_t *ids, const float *weights, const int32_t *d_slot_table,
                        int n_slots, const void *pool, size_t slot_bytes,
                        const int32_t *expert_subset, int n_subset, float *partial,
                        void *workspace, size_t ws_bytes, cudaStream_t s,
                        const moe_ffn_timing *timing);

// moe_expert_ffn_impl plus the fill sources (device [E] pinned-host image addresses of the
// experts whose slots the kernels fill while computing; NULL: none).
int moe_expert_ffn_core(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k,
                        const int32_t *ids, const float *weights, const int32_t *d_slot_table,
                        int n_slots, const void *pool, size_t slot_bytes,
                        const int32_t *expert_subset, int n_subset, const uint64_t *d_fill_src,
                        float *partial, void *workspace, size_t ws_bytes, cudaStream_t s,
                        const moe_ffn_timing *timing);

// The stages of one decode-path FFN call (T <= MOE_DECODE_MAX_T): a later stage reads what
// the earlier stages of the same call left in the workspace.
#define MOE_FFN_PERMUTE 1
#define MOE_FFN_GATEUP 2   // the gate/up GEMV
#define MOE_FFN_DOWN 4
#define MOE_FFN_REDUCE 8   // h from the gate/up kernel's K-split partial sums (no-op without a split)
#define MOE_FFN_ALL 15
// The caller guarantees that x was complete before the launch preceding this call started (so
// a gate/up launch without this call's permute kernel in front may still start early and read
// x before its dependency wait).
#define MOE_FFN_X_READY 16
// Kernels one decode-path FFN call (T <= MOE_DECODE_MAX_T, all stages) launches.
int moe_decode_ffn_launches(int T, int H, int F, int qtype, int E, int k);
int moe_expert_ffn_stages(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k,
                          const int32_t *ids, const float *weights, const int32_t *d_slot_table,
                          int n_slots, const void *pool, size_t slot_bytes,
                          const int32_t *expert_subset, int n_subset, const uint64_t *d_fill_src,
                          float *partial, void *workspace, size_t ws_bytes, cudaStream_t s,
                          const moe_ffn_timing *timing, int stages);

// Launch attributes of the decode chain's kernels: the programmatic dependency on the previous
// kernel of the stream (each kernel waits for it with griddepcontrol.wait before reading its
// outputs, so the launch and the prologue overlap the previous kernel's tail).
static inline void moe_pdl_config(cudaLaunchConfig_t *cfg, cudaLaunchAttribute *attr, dim3 grid, dim3 block,
                                  size_t smem, cudaStream_t s) {
    cfg->gridDim = grid;
    cfg->blockDim = block;
    cfg->dynamicSmemBytes = smem;
    cfg->stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
}

// Writes up to three small int32 arrays (<= 256 values each) on stream s with one launch
// (values travel as kernel parameters, so no host staging buffer outlives the call).
int moe_write_ints(int32_t *const dst[3], const int n[3], const int32_t *const src[3], cudaStream_t s);

// Pinned host image of (layer, expert) of a cache (layer global; NULL outside the group).
const void *moe_cache_image(const moe_cache *c, int layer, int expert);
// Pool base and slot count of a cache; the layer range of its group.
const void *moe_cache_pool(const moe_cache *c, int *n_slots);
int moe_cache_layer_range(const moe_cache *c, int *first_layer, int *n_layers);
bool moe_cache_is_device_managed(const moe_cache *c);

size_t moe_decode_workspace_bytes(int T, int H, int F, int qtype, int E, int k);
// moe_combine_rmsnorm skipping the routes whose id is -1 (ids [T][k] device, or NULL).
int moe_combine_rmsnorm_routes(const float *partial, const int32_t *ids, int T, int k, int H, const float *extra,
                               float *y, float *xn, float eps, cudaStream_t s);
// Workspace of moe_expert_ffn for these sizes (decode GEMV or prefill grouped GEMM path).
size_t moe_ffn_workspace_bytes(int T, int H, int F, int qtype, int xtype, int E, int k);

// Prefill path (moe_prefill.cu): grouped GEMM on tcgen05 for T > MOE_DECODE_MAX_T.
bool moe_prefill_eligible(int T, int H, int F, int qtype, int xtype);
size_t moe_prefill_workspace_bytes(int T, int H, int F, int E, int k);
int moe_prefill_ffn(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k, const int32_t *ids,
                    const float *weights, const int32_t *d_slot_table, int n_slots, const void *pool,
                    size_t slot_bytes, const int32_t *expert_subset, int n_subset, float *partial,
                    void *workspace, size_t ws_bytes, cudaStream_t s, const moe_ffn_timing *timing);

