// Prefill (batches above the decode limit): grouped GEMM on tcgen05 tensor cores.
//
// Page 4 ("llama.cpp MoE缓存实测", section "MoE缓存到底缓存了什么"): batches of more than
// 32 tokens (prompt processing) do not use the decode slots.  Here every routed token
// row is sorted by expert and each expert's FFN becomes two GEMMs over its tokens:
// [gate; up] (2F x H) times the tokens, SwiGLU, then down (H x F) times h.
//
// GB300 mapping.  The quantised weights are the operand that is dequantised, so they are
// made the MMA's M side and go to tensor memory, not shared memory:
//   D[128 weight rows][N tokens] += A[rows][K] . B[tokens][K]^T,
//   tcgen05.mma kind::f16, M = 128, N = the chunk's tokens rounded up to 16 (<= 192), K = 16,
//   A (the dequantised weights) in TMEM, B (the tokens) in shared memory, D in TMEM (fp32).
// A chunk is up to 192 tokens of one expert (an expert's tokens split into near-equal
// chunks); a work item is (chunk, 128-row weight slab).  The dequantised operand never
// passes through shared memory, and a batch with few tokens per expert runs MMAs only as
// wide as its tokens.
//  * route kernels (count, chunk, place): the routes sorted by expert into positions, the
//    chunks of every expert, experts with the most tokens first (each expert's chunks
//    consecutive, so that the items reading one expert's weights run together and share them
//    in L2);
//  * gather kernel: activations -> fp16 rows in position order (K permuted for 4-bit);
//  * GEMM kernels: persistent, one CTA per SM over a strided list of work items, warp roles
//    with mbarrier rings that run on across items:
//      warps 0, 22 per 64-column K stage (warp 0 the even stages, warp 22 the odd ones) the
//                  slab's quantised tile blocks (4-D TMA boxes over the slot pool) and the
//                  chunk's token rows (2-D TMA boxes of 64 columns x 64 rows, or one box of
//                  192 rows for a chunk of more than 128, 128-byte swizzle, straight into the
//                  UMMA layout), completing the stage's one barrier;
//      warps 2-17  four groups of four warps, group G taking the stages g = G mod 4: a thread
//                  dequantises one weight row's 64 columns — integer codes to fp16 by
//                  exponent tricks, then d*q [+ m] in one fp16 op (a single rounding) — and
//                  stores them into its group's slot of a 4-stage ring in TMEM (tcgen05.st,
//                  lane = weight row); a slot is rewritten once the MMAs of its previous
//                  stage have completed (that stage's ring release).  Every wait and hand-off
//                  costs a few hundred cycles (measured), so each role keeps several stages
//                  in flight rather than working through one stage at a time;
//      warp 1      issues the MMAs into one of two 192-column TMEM accumulators once a
//                  stage's weights are in TMEM (its group waited for the stage's copies),
//                  and one commit per stage that releases both the ring stage and the slot;
//      warps 18-21 the epilogue of the previous item from the other accumulator (lane =
//                  weight row): GEMM 1 holds 64 gate rows in lanes 0-63 and the same 64 up
//                  rows in 64-127; the up quarters pass their values through shared memory
//                  to the gate quarters, which write h = silu(g) * u as fp16 rows in position
//                  order (GEMM 2's B operand); GEMM 2 scales by the router weight and writes
//                  partial[route][rows].
//  * Operands are fp16 (activations arrive as bf16 and are rounded to fp16; bf16 operands
//    would exceed the 2e-3 output tolerance on the Qwen-shaped layer).
//  * 4-bit operands: one 32-bit word of codes decodes into the fp16 pairs (q0,q4), (q1,q5),
//    (q2,q6), (q3,q7), so inside every 8-element group of K both operands of a 4-bit GEMM
//    are stored in the order 0,4,1,5,2,6,3,7 (the same permutation of K on both sides
//    leaves the products unchanged).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_tc.cuh"

#define PF_NT 192          // most tokens of a chunk (MMA N)
#define PF_WM 128          // weight rows of a work item (MMA M)
#define PF_BK 64           // K columns per stage
#define PF_BOX_ROWS 64     // token rows per TMA box
#define PF_DQ_WARPS 16     // 4 groups of 4 (one warp per TMEM lane quarter)
#define PF_EPI_WARPS 4
#define PF_PROD2_WARP (2 + PF_DQ_WARPS + PF_EPI_WARPS)  // the producer of the odd stages
#define PF_THREADS ((PF_PROD2_WARP + 1) * 32)
#define PF_S 6             // TMA ring stages (token rows + quantised weights)
#define PF_AS 4            // TMEM ring stages of dequantised weights (32 columns each), one per
                           // dequant group
#define PF_TMEM_COLS 512   // two accumulators of PF_NT columns, then the A ring
#define PF_ACOL (2 * PF_NT)
#define PF_CTRL 13312      // control block: barriers, epilogue exchange, route lists
static_assert(PF_ACOL + PF_AS * 32 <= PF_TMEM_COLS, "TMEM budget");
static_assert(PF_S % 2 == 0, "each ring stage keeps one producer; stage pairs never wrap");
static_assert(PF_AS % 2 == 0 && PF_BK == 64, "TMEM slot pairs");
static_assert(PF_S > PF_AS, "a slot's release follows the previous fill of the stage that reuses it");
static_assert(PF_NT % 16 == 0 && PF_NT <= 256, "MMA N");

namespace {

// ------------------------------------------------------------------ workspace layout

struct PfLayout {
    int max_chunks;
    size_t o_rows, o_cexp, o_cslot, o_cpos, o_cn, o_cnt, o_cur;  // int offsets (in ints)
    size_t ints_bytes, xg, hg, total;
};

// ints[0] = chunks, ints[1] = positions placed; rows [R]: position -> route; per chunk its
// expert, slot, first position and token count; per expert its route count and placement
// cursor.
inline PfLayout pf_layout(int T, int H, int F, int E, int k) {
    PfLayout L;
    const long R = (long)T * k;
    L.max_chunks = (int)((R + PF_NT - 1) / PF_NT + E);
    size_t o = 16;
    L.o_rows = o;  o += R;
    L.o_cexp = o;  o += L.max_chunks;
    L.o_cslot = o; o += L.max_chunks;
    L.o_cpos = o;  o += L.max_chunks;
    L.o_cn = o;    o += L.max_chunks;
    L.o_cnt = o;   o += MOE_MAX_E;
    L.o_cur = o;   o += MOE_MAX_E;
    L.ints_bytes = (o * 4 + 1023) / 1024 * 1024;
    L.xg = L.ints_bytes;
    L.hg = L.xg + ((size_t)R * H * 2 + 1023) / 1024 * 1024;
    L.total = L.hg + ((size_t)R * F * 2 + 1023) / 1024 * 1024;
    return L;
}

struct PfParams {
    CUtensorMap wmap[3];  // quantised tile blocks of gate, up, down over the pool (4-D)
    CUtensorMap tmap;     // token rows: xg (GEMM 1) or hg (GEMM 2), 2-D [R][K] fp16, 64-row boxes
    CUtensorMap tmap_nt;  // the same rows in PF_NT-row boxes (one copy for a chunk of > 128 rows)
    int T, H, F, k, E;
    const float *weights;
    const int32_t *ints;
    const int32_t *rows, *c_exp, *c_slot, *c_pos, *c_n;
    __half *hg;        // GEMM 1 output (GEMM 2's token rows)
    float *partial;    // GEMM 2 output
    int *status;
};

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 4-D TMA tile load global -> shared completing on `bar`; coordinates (x, y, z, w) in elements
// of the map (x is always 0 here, so the 16-byte alignment of the innermost coordinate holds).
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int x, int y, int z, int w,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
        : "memory");
}

// 2-D TMA tile load; x (the K column) is a multiple of 64 fp16 = 128 bytes.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Shared-memory counters with release / acquire semantics at CTA scope.
__device__ __forceinline__ void red_release_add(unsigned *a, unsigned v) {
    asm volatile("red.release.cta.shared::cta.add.u32 [%0], %1;" ::"r"(smem_u32(a)), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned *a) {
    unsigned v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(a)) : "memory");
    return v;
}

// Named barrier over `count` threads.
__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier that also ANDs a predicate over the participating threads.
__device__ __forceinline__ bool named_sync_and(int id, int count, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// ------------------------------------------------------------------ route + gather

// Routes sorted by expert (restricted to a subset) into positions, in three launches over the
// whole grid: (1) per-expert route counts (shared-memory histograms, one global add per block
// and expert; ids outside [-1, E) are reported), (2) one CTA: expert offsets, the experts
// ordered by count and their chunks (below), (3) positions: each warp groups its routes by
// expert (warp match), the group's leader reserves a run of positions with one global add.
// Within an expert the order of the routes is not fixed (a route's result does not depend on
// where it sits in its chunk).
#define PF_RB 256  // threads (routes) per block of the count and place kernels

__device__ __forceinline__ int pf_expert_of(const int32_t *ids, int r, int R, int E, const int32_t *subset,
                                            int n_subset) {
    if (r >= R) return -1;
    const int v = ids[r];
    if (v < 0 || v >= E) return -1;
    if (subset) {
        bool in = false;
        for (int i = 0; i < n_subset; ++i) in |= subset[i] == v;
        if (!in) return -1;
    }
    return v;
}

__global__ void __launch_bounds__(PF_RB) pf_count_kernel(const int32_t *__restrict__ ids, int R, int E,
                                                         const int32_t *__restrict__ subset, int n_subset,
                                                         int32_t *__restrict__ cnt, int *status) {
    __shared__ int hist[MOE_MAX_E];
    for (int e = threadIdx.x; e < E; e += PF_RB) hist[e] = 0;
    __syncthreads();
    const int r = blockIdx.x * PF_RB + threadIdx.x;
    if (r < R && (ids[r] < -1 || ids[r] >= E)) moe_set_status(status, MOE_ERR_INVALID);  // -1: a dropped route
    if (subset && blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_subset; i += PF_RB)
            if (subset[i] < 0 || subset[i] >= E) moe_set_status(status, MOE_ERR_INVALID);
    const int e = pf_expert_of(ids, r, R, E, subset, n_subset);
    if (e >= 0) atomicAdd(&hist[e], 1);
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += PF_RB)
        if (hist[x]) atomicAdd(&cnt[x], hist[x]);
}

__global__ void __launch_bounds__(PF_RB) pf_place_kernel(const int32_t *__restrict__ ids, int R, int E,
                                                         const int32_t *__restrict__ subset, int n_subset,
                                                         int32_t *__restrict__ cur, int32_t *__restrict__ rows) {
    const int r = blockIdx.x * PF_RB + threadIdx.x, lane = threadIdx.x & 31;
    const int e = pf_expert_of(ids, r, R, E, subset, n_subset);
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    const int leader = __ffs(grp) - 1;
    int base = 0;
    if (e >= 0 && lane == leader) base = atomicAdd(&cur[e], __popc(grp));
    base = __shfl_sync(0xffffffffu, base, leader);
    if (e >= 0) rows[base + __popc(grp & ((1u << lane) - 1u))] = r;
}

// (2) One CTA: from the counts, the expert offsets (in id order) and placement cursors, the
// experts ordered by descending count (ties: lower id) and the chunks: an expert with c routes
// gets ceil(c / PF_NT) chunks of near-equal size (the first c % n one larger), chunk j starting
// at its expert's offset + j (c / n) + min(j, c % n), listed expert by expert in that order.
// An expert whose slot is out of range is reported and its chunks get slot -1 (skipped by the
// GEMMs).
__global__ void __launch_bounds__(1024) pf_chunk_kernel(int E, const int32_t *__restrict__ slot_table, int n_slots,
                                                        int32_t *__restrict__ ints, size_t o_cexp, size_t o_cslot,
                                                        size_t o_cpos, size_t o_cn, size_t o_cnt, size_t o_cur,
                                                        int *status) {
    __shared__ int tot[MOE_MAX_E], offs[MOE_MAX_E + 1], order[MOE_MAX_E];
    __shared__ int wsum[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cnt = tid < E ? ints[o_cnt + tid] : 0;
    if (tid < E) tot[tid] = cnt;
    {
        int x = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        int before = 0;
        for (int w = 0; w < warp; ++w) before += wsum[w];
        if (tid < E) {
            offs[tid] = before + x - cnt;
            ints[o_cur + tid] = before + x - cnt;
        }
        if (tid == E - 1) offs[E] = before + x;
    }
    __syncthreads();
    if (tid < E) {
        int rank = 0;
        for (int e = 0; e < E; ++e) rank += (tot[e] > cnt) || (tot[e] == cnt && e < tid);
        order[rank] = tid;
    }
    __syncthreads();
    const int e = tid < E ? order[tid] : -1;
    const int nch = e >= 0 ? (tot[e] + PF_NT - 1) / PF_NT : 0;
    int x = nch;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    __syncthreads();  // wsum reuse
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += wsum[w];
    if (tid == E - 1) {
        ints[0] = before + x;
        ints[1] = offs[E];
    }
    if (nch > 0) {
        int slot = slot_table ? slot_table[e] : e;
        if (slot < 0 || slot >= n_slots) {
            moe_set_status(status, MOE_ERR_INVALID);
            slot = -1;
        }
        const int c = tot[e], q = c / nch, rem = c % nch;
        const int b0 = before + x - nch;
        for (int j = 0; j < nch; ++j) {
            ints[o_cexp + b0 + j] = e;
            ints[o_cslot + b0 + j] = slot;
            ints[o_cpos + b0 + j] = offs[e] + j * q + min(j, rem);
            ints[o_cn + b0 + j] = q + (j < rem ? 1 : 0);
        }
    }
}

// Activation rows in position order -> fp16 rows (K in the 4-bit order when Q4); one warp per
// position.
template <int XT, bool Q4>
__global__ void __launch_bounds__(256) pf_gather_kernel(const void *__restrict__ x, int H, int k,
                                                        const int32_t *__restrict__ ints,
                                                        const int32_t *__restrict__ rows, __half *__restrict__ xg) {
    const int pos = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (pos >= ints[1]) return;
    const int t = rows[pos] / k;
    for (int c8 = lane; c8 < H / 8; c8 += 32) {
        const size_t base = (size_t)t * H + (size_t)c8 * 8;
        __half2 h[4];
        if (XT == MOE_BF16) {
            const uint4 raw = *(const uint4 *)((const __nv_bfloat16 *)x + base);
            const __nv_bfloat162 *b2 = (const __nv_bfloat162 *)&raw;
#pragma unroll
            for (int i = 0; i < 4; ++i) h[i] = __float22half2_rn(__bfloat1622float2(b2[i]));
        } else {
            const float4 a = *(const float4 *)((const float *)x + base);
            const float4 b = *(const float4 *)((const float *)x + base + 4);
            h[0] = __floats2half2_rn(a.x, a.y);
            h[1] = __floats2half2_rn(a.z, a.w);
            h[2] = __floats2half2_rn(b.x, b.y);
            h[3] = __floats2half2_rn(b.z, b.w);
        }
        const uint32_t *w = (const uint32_t *)h;
        uint4 v;
        if (Q4)  // (e0,e1)(e2,e3)(e4,e5)(e6,e7) -> (e0,e4)(e1,e5)(e2,e6)(e3,e7)
            v = make_uint4(__byte_perm(w[0], w[2], 0x5410), __byte_perm(w[0], w[2], 0x7632),
                           __byte_perm(w[1], w[3], 0x5410), __byte_perm(w[1], w[3], 0x7632));
        else
            v = make_uint4(w[0], w[1], w[2], w[3]);
        *(uint4 *)(xg + (size_t)pos * H + (size_t)c8 * 8) = v;
    }
}

// ------------------------------------------------------------------ dequant of 16 columns

// Raw stage layout (both GEMMs): 4 row tiles of 32 weight rows x 2 tile blocks (each the codes
// of 32 rows x 32 columns, then their 32 scale entries; slot image layout).  GEMM 1: row
// tiles 0-1 gate, 2-3 up; GEMM 2: down.
template <int QT> struct RawGeom {
    static constexpr int TBB = QT == MOE_Q8_0 ? 1088 : 640;   // bytes of a tile block
    static constexpr int SC = QT == MOE_Q8_0 ? 1024 : 512;    // its scale entries' offset
    static constexpr int BYTES = 8 * TBB;
};

__device__ __forceinline__ __half2 u32_as_half2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }
__device__ __forceinline__ uint32_t half2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// Row `lane` of raw row tile `rt`, columns 16 half .. 16 half + 15 of tile block `blk`, as 8
// fp16 pairs (TMEM columns: the A operand's K order).
//  q8_0: the offset-binary bytes q + 128 placed under the fp16 exponent of 1024 give
//        1152 + q exactly; subtracting 1152 leaves q, and one fp16 multiply by d rounds d*q
//        once.
//  4-bit: nibble pairs (n, n+4) masked under the exponent of 1024 give 1024 + q; then
//        q*d + m in one fp16 FMA (one rounding).
template <int QT>
__device__ __forceinline__ void dequant16(const uint8_t *raw, int rt, int blk, int half, int lane,
                                          uint32_t (&o)[8]) {
    using G = RawGeom<QT>;
    const uint8_t *tb = raw + (size_t)(rt * 2 + blk) * G::TBB;
    if constexpr (QT == MOE_Q8_0) {
        const __half dh = __ushort_as_half(*(const unsigned short *)(tb + G::SC + moe_scale_pos(lane) * 2));
        const __half2 d2 = __halves2half2(dh, dh);
        const __half2 off = __float2half2_rn(1152.0f);
        const uint4 q = *(const uint4 *)(tb + moe_piece_in_block(half, lane));
        const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 lo = __hsub2(u32_as_half2(__byte_perm(wd[i], 0x64646464u, 0x4140)), off);
            const __half2 hi = __hsub2(u32_as_half2(__byte_perm(wd[i], 0x64646464u, 0x4342)), off);
            o[2 * i] = half2_as_u32(__hmul2(lo, d2));
            o[2 * i + 1] = half2_as_u32(__hmul2(hi, d2));
        }
    } else {
        const uint32_t dm = *(const uint32_t *)(tb + G::SC + moe_scale_pos(lane) * 4);
        const uint2 q = *(const uint2 *)(tb + moe_piece_in_block(0, lane) + 8 * half);
        const __half dh = __ushort_as_half((unsigned short)(dm & 0xFFFFu));
        const __half mh = __ushort_as_half((unsigned short)(dm >> 16));
        const __half2 d2 = __halves2half2(dh, dh), m2 = __halves2half2(mh, mh);
        const __half2 off = __float2half2_rn(1024.0f);
        const uint32_t wd[2] = {q.x, q.y};
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const uint32_t u = ((wd[i] >> (4 * n)) & 0x000F000Fu) | 0x64006400u;
                o[4 * i + n] = half2_as_u32(__hfma2(__hsub2(u32_as_half2(u), off), d2, m2));
            }
    }
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    const uint32_t a = smem_u32(p);
    return p + ((1024 - (a & 1023)) & 1023);
}

// Wait for an mbarrier phase; gives up (returns false) when another role has aborted or,
// after the spin limit, records MOE_ERR_TIMEOUT and aborts the CTA.  It polls with the
// non-blocking test (measured: a try_wait that suspends the thread adds hundreds of cycles
// to every hand-off between the roles).
__device__ __forceinline__ bool pf_wait(uint64_t *bar, uint32_t parity, int *status, volatile int *abort_flag) {
    for (uint32_t i = 0; i < MOE_TEST_SPIN_LIMIT; ++i) {
        if (mbar_test_wait(bar, parity)) return true;
        if (*abort_flag) return false;
    }
    moe_set_status(status, MOE_ERR_TIMEOUT);
    *abort_flag = 1;
    return false;
}

// ------------------------------------------------------------------ the persistent GEMM

template <int QT>
struct PfGeom {
    static constexpr int TOKB = PF_NT * 128;                  // token rows of a stage (64 fp16 each)
    static constexpr int STAGE = ((TOKB + RawGeom<QT>::BYTES) + 1023) / 1024 * 1024;
    static constexpr size_t SMEM = 1024 + PF_CTRL + (size_t)PF_S * STAGE;
};

// Work item j = (chunk j / MT, weight slab j % MT); CTA c takes j = c, c+G, ...
// GEMM 1 (DOWN = false): slab m = gate rows 64m.. (TMEM lanes 0-63) and up rows 64m.. (lanes
// 64-127) of F x H against the chunk's x rows; epilogue h = silu(g) * u -> fp16 rows of hg.
// GEMM 2: slab m = down rows 128m.. of H x F against h; epilogue w[r] * (.) -> partial[r].
template <int QT, bool DOWN>
__global__ void __launch_bounds__(PF_THREADS, 1) pf_gemm_kernel(const __grid_constant__ PfParams p) {
    extern __shared__ uint8_t smem_raw[];
    using G = RawGeom<QT>;
    using PG = PfGeom<QT>;
    const int MT = DOWN ? p.H / PF_WM : p.F / 64;
    const int NK = (DOWN ? p.F : p.H) / PF_BK;
    const int n_items = p.ints[0] * MT;
    if ((int)blockIdx.x >= n_items) return;

    uint8_t *smem = align1024(smem_raw);
    uint64_t *s_full = (uint64_t *)smem;
    uint64_t *s_empty = s_full + PF_S;
    uint64_t *acc_full = s_empty + PF_S;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *mma_done = acc_empty + 2;
    uint32_t *tmem_slot = (uint32_t *)(mma_done + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    unsigned *a_cnt = (unsigned *)(smem + 512);  // per TMEM slot pair: dequant warps done (monotonic)
    float *xch = (float *)(smem + 1024);              // [2 pairs][2 slots][32 lanes][16] (GEMM 1)
    int *e_route = (int *)(smem + 1024 + 8192);       // [2 accumulators][PF_NT] (GEMM 2)
    float *e_w = (float *)(e_route + 2 * PF_NT);
    uint8_t *ring = smem + PF_CTRL;
    static_assert(1024 + 8192 + 2 * PF_NT * 8 <= PF_CTRL && PF_CTRL % 1024 == 0, "control block");

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < PF_S; ++s) {
            mbar_init(&s_full[s], 1);  // the stage's producer
            mbar_init(&s_empty[s], 1);
        }
        for (int s = 0; s < PF_AS; ++s) a_cnt[s] = 0;
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], PF_EPI_WARPS);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, PF_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 || warp == PF_PROD2_WARP) {
        // ---------------- producers (lane 0): warp 0 the even K stages, the last warp the odd
        // ones (PF_S is even, so each ring stage always has the same producer); per stage the
        // chunk's token rows and the slab's quantised tile blocks.  A one-thread loop is bound
        // by its own instruction latency (measured: a few hundred cycles per wait or copy
        // issue), so two of them share the stages; each keeps its stage index and phase in
        // registers (no division per stage).
        if (lane == 0) {
            const uint32_t mine = warp == 0 ? 0u : 1u;
            int g = 0;
            uint32_t s = 0, ph = 0;  // ring stage of stage g, and the parity of its last release
            bool ok = true;
            for (int j = blockIdx.x; j < n_items && ok; j += gridDim.x) {
                const int c = j / MT, m = j % MT;
                const int slot = p.c_slot[c];
                if (slot < 0) continue;
                const int pos0 = p.c_pos[c], n = p.c_n[c];
                // a chunk of more than 128 rows comes in one PF_NT-row box, a smaller one in
                // 64-row boxes (rows past the chunk belong to the next one or read 0: unused)
                const bool big = n > 2 * PF_BOX_ROWS;
                const int nbox = big ? 1 : (n + PF_BOX_ROWS - 1) / PF_BOX_ROWS;
                const uint32_t bytes =
                    (big ? (uint32_t)PF_NT * 128u : (uint32_t)(nbox * PF_BOX_ROWS * 128)) + (uint32_t)G::BYTES;
                uint8_t *st = ring + (size_t)s * PG::STAGE;
                for (int kc = 0; kc < NK; ++kc, ++g) {
                    if ((s & 1u) == mine) {
                        if (g >= PF_S && !(ok = pf_wait(&s_empty[s], ph ^ 1u, p.status, abort_flag))) break;
                        mbar_arrive_expect_tx(&s_full[s], bytes);
                        if (big) {
                            tma_load_2d(st, &p.tmap_nt, kc * PF_BK, pos0, &s_full[s]);
                        } else {
                            for (int b = 0; b < nbox; ++b)
                                tma_load_2d(st + b * PF_BOX_ROWS * 128, &p.tmap, kc * PF_BK, pos0 + PF_BOX_ROWS * b,
                                            &s_full[s]);
                        }
                        if (DOWN) {
                            tma_load_4d(st + PG::TOKB, &p.wmap[2], 0, 2 * kc, 4 * m, slot, &s_full[s]);
                        } else {
                            tma_load_4d(st + PG::TOKB, &p.wmap[0], 0, 2 * kc, 2 * m, slot, &s_full[s]);
                            tma_load_4d(st + PG::TOKB + 4 * G::TBB, &p.wmap[1], 0, 2 * kc, 2 * m, slot, &s_full[s]);
                        }
                    }
                    if (++s == PF_S) {
                        s = 0;
                        ph ^= 1u;
                        st = ring;
                    } else {
                        st += PG::STAGE;
                    }
                }
            }
            // never leave with copies in flight: wait for the last phase issued on each of this
            // producer's stages
            for (int q = (int)mine; q < PF_S && q < g; q += 2) {
                const int last = q + ((g - 1 - q) / PF_S) * PF_S;
                mbar_wait_bounded(&s_full[q], (last / PF_S) & 1, p.status);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (lane 0).  Its loop is the kernel's critical path: a chain
        // of dependent instructions (measured: ~45 clocks per tcgen05 instruction issued and ~5
        // per dependent ALU instruction), so it takes the K stages two at a time (one acquire
        // and one fence per pair, eight MMAs), and carries the stage and slot indexes, the
        // descriptors and the dequant count a slot pair needs in registers.  NK is even (the
        // host requires H and F to be multiples of 128), so a pair never straddles two items,
        // and g is even at every pair: the pair's slots are {0, 1} or {2, 3}, its ring stages
        // s and s + 1 (PF_S is even).
        if (lane == 0) {
            int jl = 0;
            bool ok = true;
            uint32_t s = 0, sph = 0;    // ring stage of the pair's first stage, parity of its fill
            uint32_t pc = 0, want = 8;  // slot pair, and the dequant count its next use needs
            const uint64_t b_first = umma_desc_sw128(smem_u32(ring));
            uint64_t b = b_first;
            uint32_t a = tmem + PF_ACOL;
            for (int j = blockIdx.x; j < n_items && ok; j += gridDim.x) {
                const int c = j / MT;
                if (p.c_slot[c] < 0) continue;
                const uint32_t npad = (uint32_t)(p.c_n[c] + 15) & ~15u;
                const uint32_t idesc = umma_idesc_f16_f32(PF_WM, (int)npad);
                const int buf = jl & 1;
                if (jl >= 2 && !(ok = pf_wait(&acc_empty[buf], ((jl / 2) - 1) & 1, p.status, abort_flag))) break;
                tc_fence_after();
                const uint32_t d = tmem + buf * PF_NT;
                for (int kc = 0; kc < NK; kc += 2) {
                    // both stages' weights are in TMEM once their two dequant groups' eight warps
                    // counted themselves in (release / acquire on the pair's shared counter)
                    if (ld_acquire(&a_cnt[pc]) < want) {
                        uint32_t i = 0;
                        while (ld_acquire(&a_cnt[pc]) < want) {
                            if (++i >= MOE_TEST_SPIN_LIMIT) {
                                moe_set_status(p.status, MOE_ERR_TIMEOUT);
                                *abort_flag = 1;
                            }
                            if (*abort_flag) {
                                ok = false;
                                break;
                            }
                        }
                        if (!ok) break;
                    }
                    // the tokens the MMAs read were landed by TMA: observe both fills here too (they
                    // completed before the dequant groups counted in, so the tests pass at once)
                    if (!mbar_test_wait(&s_full[s], sph) && !(ok = pf_wait(&s_full[s], sph, p.status, abort_flag)))
                        break;
                    if (!mbar_test_wait(&s_full[s + 1], sph) &&
                        !(ok = pf_wait(&s_full[s + 1], sph, p.status, abort_flag)))
                        break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < PF_BK / 16; ++kk)
                        umma_f16_tmem_a(d, a + 8 * kk, b + 2 * kk, idesc, (kc > 0 || kk > 0) ? 1u : 0u);
                    // one commit per stage frees the ring stage (producers) and its TMEM slot (the
                    // dequant group that next writes the slot waits for this stage's release)
                    umma_commit(&s_empty[s]);
                    const uint64_t b2 = b + (PG::STAGE >> 4);
#pragma unroll
                    for (int kk = 0; kk < PF_BK / 16; ++kk)
                        umma_f16_tmem_a(d, a + 32 + 8 * kk, b2 + 2 * kk, idesc, 1u);
                    umma_commit(&s_empty[s + 1]);
                    if ((s += 2) == PF_S) {
                        s = 0;
                        sph ^= 1u;
                        b = b_first;
                    } else {
                        b = b2 + (PG::STAGE >> 4);
                    }
                    if (++pc == PF_AS / 2) {
                        pc = 0;
                        want += 8;
                        a = tmem + PF_ACOL;
                    } else {
                        a += 64;
                    }
                }
                if (ok) umma_commit(&acc_full[buf]);
                ++jl;
            }
            // every MMA of this CTA has completed before TMEM is released
            umma_commit(mma_done);
            mbar_wait_bounded(mma_done, 0, p.status);
        }
    } else if (warp < 2 + PF_DQ_WARPS) {
        // ---------------- dequant: group dg = (warp - 2) / 4 takes the stages g = dg mod 4 and
        // TMEM slot dg; warp -> TMEM lane quarter q = warp % 4 = raw row tile q; thread -> one
        // weight row, all 64 columns of the stage
        const int q = warp & 3, dg = (warp - 2) >> 2;
        const uint32_t a_addr = tmem + ((uint32_t)(32 * q) << 16) + PF_ACOL + 32 * dg;
        int g = 0;
        bool ok = true;
        for (int j = blockIdx.x; j < n_items && ok; j += gridDim.x) {
            if (p.c_slot[j / MT] < 0) continue;
            for (int kc = 0; kc < NK; ++kc, ++g) {
                if ((g & (PF_AS - 1)) != dg) continue;
                const int s = g % PF_S;
                bool w = true;
                if (lane == 0) {
                    // The TMEM slot is free once the MMAs of stage g - PF_AS (its previous use) have
                    // completed: that stage's ring release.  It is waited for first: a group sees
                    // only every other fill of a ring stage (stage g - PF_S belongs to another
                    // group), and a parity test cannot tell the fill of stage g from that earlier
                    // one while the earlier one is still landing.  The release of g - PF_AS comes
                    // after the MMA issuer saw the fill of g - PF_S, so after it the parity of
                    // s_full[s] can only mean stage g.
                    if (g >= PF_AS)
                        w = pf_wait(&s_empty[(g - PF_AS) % PF_S], ((g - PF_AS) / PF_S) & 1, p.status, abort_flag);
                    if (w) w = pf_wait(&s_full[s], (g / PF_S) & 1, p.status, abort_flag);
                }
                w = __shfl_sync(0xffffffffu, w, 0);
                if (!(ok = w)) break;  // the warp leaves together
                // every lane observes both completed phases itself (one test each), so that each
                // lane's reads of the stage and writes of the slot are ordered after them
                if (g >= PF_AS) mbar_test_wait(&s_empty[(g - PF_AS) % PF_S], ((g - PF_AS) / PF_S) & 1);
                mbar_test_wait(&s_full[s], (g / PF_S) & 1);
                tc_fence_after();
                uint32_t o[32];
                const uint8_t *raw = ring + (size_t)s * PG::STAGE + PG::TOKB;
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    dequant16<QT>(raw, q, h >> 1, h & 1, lane, *reinterpret_cast<uint32_t(*)[8]>(&o[8 * h]));
                tmem_st32(a_addr, o);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) red_release_add(&a_cnt[dg >> 1], 1);  // the slot pair's counter
            }
        }
    } else if (warp < PF_PROD2_WARP) {
        // ---------------- epilogue: TMEM lane quarter q = warp % 4, lane = weight row 32 q + lane
        const int q = warp & 3, ew = warp - 2 - PF_DQ_WARPS;
        int jl = 0, xs = 0;  // items done, exchange chunks done (slot parity)
        bool ok = true;
        for (int j = blockIdx.x; j < n_items && ok; j += gridDim.x) {
            const int c = j / MT, m = j % MT;
            if (p.c_slot[c] < 0) continue;
            const int pos0 = p.c_pos[c], n = p.c_n[c];
            const int buf = jl & 1;
            if (DOWN)  // this chunk's routes and router weights, read before the accumulator is ready
                for (int i = ew * 32 + lane; i < n; i += 32 * PF_EPI_WARPS) {
                    const int r = p.rows[pos0 + i];
                    e_route[buf * PF_NT + i] = r;
                    e_w[buf * PF_NT + i] = p.weights[r];
                }
            const bool w = ew == 0 && lane == 0 ? pf_wait(&acc_full[buf], (jl / 2) & 1, p.status, abort_flag) : true;
            // one thread waited; the four epilogue warps agree (and the route lists are written)
            // before going on
            if (!(ok = named_sync_and(1, 32 * PF_EPI_WARPS, w))) break;
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16) + buf * PF_NT;
            for (int c0 = 0; c0 < n; c0 += 16, ++xs) {
                uint32_t v[16];
                tmem_ld16(tb + c0, v);
                tmem_ld_wait();
                const int nn = min(16, n - c0);
                if (!DOWN) {
                    // up quarters (2, 3) hand their values to the gate quarters (0, 1); column i of
                    // lane l at xb[32 i + l] (no bank conflicts)
                    float *xb = xch + (size_t)((q & 1) * 2 + (xs & 1)) * 512 + lane;
                    if (q >= 2)
#pragma unroll
                        for (int i = 0; i < 16; ++i) xb[32 * i] = __uint_as_float(v[i]);
                    named_sync(2 + (q & 1), 64);
                    if (q < 2) {
                        const int f = 64 * m + 32 * q + lane;
                        const int fp = QT == MOE_Q4_SM ? (f & ~7) + (f & 3) * 2 + ((f >> 2) & 1) : f;
                        __half *dst = p.hg + (size_t)(pos0 + c0) * p.F + fp;
                        // every shared-memory load first (one round trip), then all 16 values
                        // computed side by side (no per-column branch: 16 independent chains), then
                        // the stores
                        __half hv[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float gv = __uint_as_float(v[i]);
                            hv[i] = __float2half_rn(__fdividef(gv, 1.0f + __expf(-gv)) * xb[32 * i]);
                        }
                        if (nn == 16) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) dst[(size_t)i * p.F] = hv[i];
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                if (i < nn) dst[(size_t)i * p.F] = hv[i];
                        }
                    }
                } else {
                    const int hr = PF_WM * m + 32 * q + lane;
                    // every shared-memory load first (one round trip), then the stores
                    int rt[16];
                    float wt[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        rt[i] = e_route[buf * PF_NT + c0 + i];
                        wt[i] = e_w[buf * PF_NT + c0 + i];
                    }
                    if (nn == 16) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) p.partial[(size_t)rt[i] * p.H + hr] = wt[i] * __uint_as_float(v[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (i < nn) p.partial[(size_t)rt[i] * p.H + hr] = wt[i] * __uint_as_float(v[i]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
            ++jl;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, PF_TMEM_COLS);
    }
}

// cuTensorMapEncodeTiled from the driver (looked up once through the runtime).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
    });
    return fn;
}

// Map of one matrix (mat: 0 gate, 1 up, 2 down) of every slot: tile blocks as [slot][row
// tile][block][TBB / 8 x uint64]; boxes of 2 K blocks x `tiles` row tiles.
template <int QT>
int encode_matrix_map(const uint8_t *pool, int n_slots, size_t slot_bytes, int H, int F, int mat, int tiles,
                      CUtensorMap *map) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return MOE_ERR_UNSUPPORTED;
    using G = RawGeom<QT>;
    const int R = mat == 2 ? H : F, K = mat == 2 ? F : H;
    const int NB = K / 32;
    const uint8_t *base = pool + moe_expert_matrix_offset(QT, H, F, mat);
    const cuuint64_t dims[4] = {(cuuint64_t)(G::TBB / 8), (cuuint64_t)NB, (cuuint64_t)(R / 32), (cuuint64_t)n_slots};
    const cuuint64_t strides[3] = {(cuuint64_t)G::TBB, (cuuint64_t)NB * G::TBB, (cuuint64_t)slot_bytes};
    const cuuint32_t box[4] = {(cuuint32_t)(G::TBB / 8), 2, (cuuint32_t)tiles, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 4, (void *)base, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

// Map of fp16 token rows [rows][K] (row stride K): boxes of 64 columns x box_rows rows with the
// 128-byte swizzle, which lands them in the UMMA K-major layout; rows past the end read 0.
int encode_rows_map(const __half *base, int rows, int K, int box_rows, CUtensorMap *map) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return MOE_ERR_UNSUPPORTED;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {PF_BK, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    if (enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (void *)base, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

// SM count of the current device, looked up once per device.
int sm_count_cached() {
    static std::mutex mu;
    static int n[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    std::lock_guard<std::mutex> lock(mu);
    if (!n[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
        n[dev] = v;
    }
    return n[dev];
}

// The GEMMs' dynamic shared-memory limit, raised once per device.
template <int QT>
int pf_set_smem_attr() {
    static std::mutex mu;
    static bool done[64] = {false};
    int dev = -1;
    MOE_TRY_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
        MOE_TRY_CUDA(cudaFuncSetAttribute(pf_gemm_kernel<QT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)PfGeom<QT>::SMEM));
        MOE_TRY_CUDA(cudaFuncSetAttribute(pf_gemm_kernel<QT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)PfGeom<QT>::SMEM));
        done[dev] = true;
    }
    return MOE_OK;
}

template <int QT>
int launch_gemms(PfParams &p1, PfParams &p2, int max_chunks, cudaStream_t s, const moe_ffn_timing *timing) {
    using PG = PfGeom<QT>;
    if (PG::SMEM > 227 * 1024) return MOE_ERR_UNSUPPORTED;
    const int rc = pf_set_smem_attr<QT>();
    if (rc != MOE_OK) return rc;
    const int sms = sm_count_cached();
    const int items1 = max_chunks * (p1.F / 64), items2 = max_chunks * (p1.H / PF_WM);
    if (timing && timing->gateup0) MOE_TRY_CUDA(cudaEventRecord(timing->gateup0, s));
    pf_gemm_kernel<QT, false><<<std::min(items1, sms), PF_THREADS, PG::SMEM, s>>>(p1);
    MOE_TRY_CUDA(cudaGetLastError());
    if (timing && timing->gateup1) MOE_TRY_CUDA(cudaEventRecord(timing->gateup1, s));
    if (timing && timing->down0) MOE_TRY_CUDA(cudaEventRecord(timing->down0, s));
    pf_gemm_kernel<QT, true><<<std::min(items2, sms), PF_THREADS, PG::SMEM, s>>>(p2);
    MOE_TRY_CUDA(cudaGetLastError());
    if (timing && timing->down1) MOE_TRY_CUDA(cudaEventRecord(timing->down1, s));
    return MOE_OK;
}

}  // namespace

bool moe_prefill_eligible(int T, int H, int F, int qtype, int xtype) {
    return T > MOE_DECODE_MAX_T && xtype == MOE_BF16 && H % 128 == 0 && F % 128 == 0 &&
           (qtype == MOE_Q8_0 || qtype == MOE_Q4_SM);
}

size_t moe_prefill_workspace_bytes(int T, int H, int F, int E, int k) { return pf_layout(T, H, F, E, k).total; }

int moe_prefill_ffn(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k, const int32_t *ids,
                    const float *weights, const int32_t *d_slot_table, int n_slots, const void *pool,
                    size_t slot_bytes, const int32_t *expert_subset, int n_subset, float *partial,
                    void *workspace, size_t ws_bytes, cudaStream_t s, const moe_ffn_timing *timing) {
    const PfLayout L = pf_layout(T, H, F, E, k);
    MOE_CHECK(ws_bytes >= L.total);
    const int R = T * k;
    PfParams p;
    p.T = T; p.H = H; p.F = F; p.k = k; p.E = E;
    p.weights = weights;
    int32_t *ints = (int32_t *)workspace;
    p.ints = ints;
    p.rows = ints + L.o_rows;
    p.c_exp = ints + L.o_cexp;
    p.c_slot = ints + L.o_cslot;
    p.c_pos = ints + L.o_cpos;
    p.c_n = ints + L.o_cn;
    __half *xg = (__half *)((uint8_t *)workspace + L.xg);
    p.hg = (__half *)((uint8_t *)workspace + L.hg);
    p.partial = partial;
    p.status = moe_status_word_device_ptr();
    const bool q8 = qtype == MOE_Q8_0;
    for (int mat = 0; mat < 3; ++mat) {
        const int tiles = mat == 2 ? 4 : 2;
        const int rc = q8 ? encode_matrix_map<MOE_Q8_0>((const uint8_t *)pool, n_slots, slot_bytes, H, F, mat, tiles,
                                                        &p.wmap[mat])
                          : encode_matrix_map<MOE_Q4_SM>((const uint8_t *)pool, n_slots, slot_bytes, H, F, mat,
                                                         tiles, &p.wmap[mat]);
        if (rc != MOE_OK) return rc;
    }
    PfParams p2 = p;
    int rc = encode_rows_map(xg, R, H, PF_BOX_ROWS, &p.tmap);
    if (rc == MOE_OK) rc = encode_rows_map(xg, R, H, PF_NT, &p.tmap_nt);
    if (rc == MOE_OK) rc = encode_rows_map(p.hg, R, F, PF_BOX_ROWS, &p2.tmap);
    if (rc == MOE_OK) rc = encode_rows_map(p.hg, R, F, PF_NT, &p2.tmap_nt);
    if (rc != MOE_OK) return rc;

    if (timing && timing->permute0) MOE_TRY_CUDA(cudaEventRecord(timing->permute0, s));
    const int rblocks = (R + PF_RB - 1) / PF_RB;
    MOE_TRY_CUDA(cudaMemsetAsync(ints + L.o_cnt, 0, MOE_MAX_E * sizeof(int32_t), s));
    pf_count_kernel<<<rblocks, PF_RB, 0, s>>>(ids, R, E, expert_subset, n_subset, ints + L.o_cnt, p.status);
    MOE_TRY_CUDA(cudaGetLastError());
    pf_chunk_kernel<<<1, 1024, 0, s>>>(E, d_slot_table, n_slots, ints, L.o_cexp, L.o_cslot, L.o_cpos, L.o_cn, L.o_cnt,
                                       L.o_cur, p.status);
    MOE_TRY_CUDA(cudaGetLastError());
    pf_place_kernel<<<rblocks, PF_RB, 0, s>>>(ids, R, E, expert_subset, n_subset, ints + L.o_cur, ints + L.o_rows);
    MOE_TRY_CUDA(cudaGetLastError());
    const int gblocks = (R + 7) / 8;
    const bool q4 = !q8;
    if (xtype == MOE_BF16) {
        if (q4) pf_gather_kernel<MOE_BF16, true><<<gblocks, 256, 0, s>>>(x, H, k, ints, p.rows, xg);
        else pf_gather_kernel<MOE_BF16, false><<<gblocks, 256, 0, s>>>(x, H, k, ints, p.rows, xg);
    } else {
        if (q4) pf_gather_kernel<MOE_F32, true><<<gblocks, 256, 0, s>>>(x, H, k, ints, p.rows, xg);
        else pf_gather_kernel<MOE_F32, false><<<gblocks, 256, 0, s>>>(x, H, k, ints, p.rows, xg);
    }
    MOE_TRY_CUDA(cudaGetLastError());
    if (timing && timing->permute1) MOE_TRY_CUDA(cudaEventRecord(timing->permute1, s));
    return q8 ? launch_gemms<MOE_Q8_0>(p, p2, L.max_chunks, s, timing)
              : launch_gemms<MOE_Q4_SM>(p, p2, L.max_chunks, s, timing);
}
