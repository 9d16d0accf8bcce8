// Decode-time expert FFN: permute (P1), gate/up dequantising GEMV with SwiGLU (G1), down
// GEMV with the router-weighted scatter (G2), combine (C1).
//
// What is computed (pages 1-5, see moe.h): for every route (t, j) of a token t to its
// j-th selected expert e, h = silu(Wg_e x_t) * (Wu_e x_t) and
// partial[t][j] = w[t][j] * (Wd_e h); the combine sums partial over j.  Weights stay in
// their quantised blocks (page 5, section 1.2) and are dequantised in registers.
//
// GB300 mapping (the decode GEMVs stream the selected experts' bytes from HBM once):
//  * the routes of an expert are cut into groups of at most 4 ("virtual experts");
//    a work unit is NTL 32-row tiles of one virtual expert over a K range: the gate and the
//    up tile of the same rows (G1), or one or two neighbouring down tiles (G2);
//  * persistent CTAs of 16 warps, one per SM, each over a contiguous range of units of equal
//    count (precomputed by the permute kernel; in the gate/up launch each CTA keeps to one K
//    range, so it stages x before its dependency wait).  The warps of a CTA take its units in
//    turn and are independent: each has its own ring of shared-memory stages, filled a few
//    chunks ahead by bulk copies (TMA engine, cp.async.bulk, issued by lane 0) or, for a
//    missed expert, by cp.async pieces from its pinned host image, and waits on its own
//    mbarriers.  There is no block-wide barrier while weights stream;
//  * a warp owns whole rows of its unit and needs no reduction with other warps: the codes
//    of a 32-column block are turned into fp16 (exact small integers) in registers, laid
//    out directly as the A fragments of mma.sync m16n8k16 (rows = weight rows, columns =
//    tokens, fp32 accumulation), and the block's fp32 scale is applied to the block's
//    partial sums in fp32, so the per-block arithmetic is exact except for the activations;
//  * activations enter the tensor core as fp16 hi + lo parts of a per-token power-of-two
//    scaled copy (about 22 significant bits), staged in shared memory for all warps of the
//    CTA: once per CTA (x over its K range, G1) or per virtual expert (h rows, G2);
//  * the warp's epilogue forms h = silu(gate) * up (G1, whole K) or stores the two partial
//    sums (G1, K split; a small kernel between the GEMVs sums them in K order and forms h),
//    or writes w[r] * (Wd h) for each route r (G2);
//  * an expert that missed in a device-managed pool is read from its pinned host image over
//    the CPU-GPU link into the ring and written through from there to its slot by the warps
//    that use the bytes ("fill" chunks).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "moe_ptx.cuh"

#define GV_WARPS 16
#define GV_THREADS (GV_WARPS * 32)
#define GV_TOK 4                  // routes of a virtual expert (one m16n8 column set: hi + lo)
#define GV_SMEM_MAX (220 * 1024)  // dynamic shared memory a GEMV kernel may take
#define GV_BARS 2048              // mbarriers: a gate/up and a down set of GV_WARPS x GV_MAX_STAGES
#define GV_MAX_STAGES 8           // ring stages of one warp
#define GV_MIN_STAGES 2
#define GV_CHUNK_TARGET 5120      // bytes of one ring stage (a chunk of a unit)
#define GV_MAX_GRID 1024          // CTAs per launch (bounds the precomputed range tables)
#define GV_UNITS_TARGET 1824      // units per launch the K split aims for (~12 per CTA)
#define GV_KS_MAX 8               // largest K split of the gate/up GEMV
#define GV_ACT_SLOTS_MAX 3        // staged (virtual expert, K range) pairs per CTA phase
#define GV_PHASE_PAIRS 64         // pairs (used or skipped) per CTA phase
#define GV_PERMUTE_MAX_R (MOE_DECODE_MAX_T * MOE_MAX_K)  // routes of one decode call

namespace {

// ------------------------------------------------------------------ launch plan

// Per kernel: NTL tiles per unit, nbr 32-column blocks per unit (the K range), CB blocks per
// chunk (one ring stage), the staged activation slot of one (virtual expert, K range) pair
// and how many of those a CTA phase holds, and the ring bytes left for the warps.
struct GvGeom {
    int NTL, nbr, CB, chunk_bytes, slot_bytes, act_slots, ring_bytes;
};

struct GvPlan {
    int KS, TPU;
    GvGeom g1, g2;
};

__host__ __device__ inline int gv_qb(int qtype) { return qtype == MOE_Q8_0 ? 1024 : 512; }  // codes / block / tile
__host__ __device__ inline int gv_sb(int qtype) { return 32 * moe_scale_entry_bytes(qtype); }

// Row stride of the staged fp16 activations (bytes): 2 Kr + 32 keeps 16-byte alignment
// and spreads the 8 rows of a B-fragment load over the banks.
// Row stride of a staged activation row (fp16, Kr columns): a multiple of 128 bytes, so that
// every hi row starts on bank 0, with room for a lo row to start 64 bytes (16 banks) into its
// row.  The eight lanes of one phase of a 16-byte shared-memory load read one route's hi and
// lo rows (B columns 2 s and 2 s + 1, below), which therefore fall on opposite halves of the
// banks whatever the route's token is: no bank conflicts.
#define GV_LO_SHIFT 64
__host__ __device__ inline int gv_row_stride(int Kr) { return (2 * Kr + GV_LO_SHIFT + 127) / 128 * 128; }

// One pair's slot: 2*NTS fp16 rows (hi, lo per token row), up to 32 inverse token scales,
// the header (SlotHdr, 128 bytes), and for the 4-bit format the per-block activation sums
// [nbr][NTS].  The gate/up kernel stages every token of the call (NTS = T <= 32), the down
// kernel the routes of one virtual expert (NTS = GV_TOK).
#define GV_INV_OFF(NTS, RS) ((size_t)2 * (NTS) * (RS))
#define GV_HDR_OFF(NTS, RS) ((size_t)2 * (NTS) * (RS) + 128)
#define GV_ASUM_OFF(NTS, RS) ((size_t)2 * (NTS) * (RS) + 256)
#define GV_SLOT_MAX (72 * 1024)  // the gate/up K split is raised until a slot fits
__host__ __device__ inline int gv_slot_bytes(int qtype, int nbr, int NTS) {
    const int b = (int)GV_ASUM_OFF(NTS, gv_row_stride(nbr * 32)) + (qtype == MOE_Q4_SM ? nbr * NTS * 4 : 0);
    return (b + 127) / 128 * 128;
}

inline bool gv_geom(int qtype, int NTL, int nbr, int NTS, GvGeom *g) {
    g->NTL = NTL;
    g->nbr = nbr;
    const int per_block = NTL * (gv_qb(qtype) + gv_sb(qtype));
    g->CB = std::max(1, std::min(nbr, GV_CHUNK_TARGET / per_block));
    g->chunk_bytes = g->CB * per_block;
    g->slot_bytes = gv_slot_bytes(qtype, nbr, NTS);
    const int ring_min = GV_WARPS * GV_MIN_STAGES * g->chunk_bytes;
    const int room = GV_SMEM_MAX - GV_BARS - ring_min;
    if (room < g->slot_bytes) return false;
    g->act_slots = std::min(GV_ACT_SLOTS_MAX, room / g->slot_bytes);
    g->ring_bytes = GV_SMEM_MAX - GV_BARS - g->act_slots * g->slot_bytes;
    return true;
}

inline int gv_smem_bytes(const GvGeom &g) { return GV_BARS + g.ring_bytes + g.act_slots * g.slot_bytes; }

// The gate/up K split is the smallest power of two giving about GV_UNITS_TARGET units (at
// most GV_KS_MAX, each K range at least one block); the down kernel takes two row tiles per
// unit when that still gives enough units.
inline bool gv_plan(int T, int H, int F, int qtype, int n_act_max, GvPlan *pl) {
    if (T < 1 || T > MOE_DECODE_MAX_T) return false;
    const int NB = H / 32, RTF = F / 32, RTH = H / 32;
    int ks = 1;
    while (ks < GV_KS_MAX && (long)n_act_max * RTF * ks < GV_UNITS_TARGET && NB % (2 * ks) == 0) ks *= 2;
    while (gv_slot_bytes(qtype, NB / ks, T) > GV_SLOT_MAX && NB % (2 * ks) == 0 && ks < 16) ks *= 2;
    // and until the staged activations fit beside the smallest ring (4-bit blocks leave less
    // room: at hidden 2048 and 32 tokens the slot of a 2-way split does not fit)
    while (!gv_geom(qtype, 2, NB / ks, T, &pl->g1) && NB % (2 * ks) == 0 && ks < 16) ks *= 2;
    pl->KS = ks;
    pl->TPU = RTH % 2 == 0 && (long)n_act_max * (RTH / 2) >= GV_UNITS_TARGET ? 2 : 1;
    return gv_geom(qtype, 2, NB / ks, T, &pl->g1) && gv_geom(qtype, pl->TPU, F / 32, GV_TOK, &pl->g2);
}

inline int gv_n_act_max(int T, int E, int k) { return T * k < E ? T * k : E; }
// virtual experts: at most one per active expert plus one per further group of GV_TOK routes
inline int gv_n_virt_max(int T, int E, int k) { return gv_n_act_max(T, E, k) + (T * k) / GV_TOK + 1; }

// ------------------------------------------------------------------ workspace layout

// Per virtual expert, written by the permute kernel.
struct ActInfo {
    unsigned long long src;  // image base the weights are read from (slot, or pinned host image)
    unsigned long long dst;  // slot base (written through when wt != 0)
    int pos0, n_e;           // route positions [pos0, pos0 + n_e); n_e == 0: skip (invalid slot)
    int fill, wt;            // fill: read src with loads (host image); wt: write the bytes to dst
    int rt[GV_TOK];          // the routes t*k + j at those positions
};

// Header of a staged slot: the pair's virtual expert and, for the down kernel, its routes'
// router weights.
struct SlotHdr {
    ActInfo in;
    float w[GV_TOK];
};
static_assert(sizeof(SlotHdr) <= 128, "slot header");

// ints[GV_SYNC_OFF], [GV_SYNC_OFF + 1]: the fused GEMV launch's grid barrier (count, generation)
#define GV_SYNC_OFF 4
// int32 region: [0] n_active [1] n_virtual | active [E] | a_off [E+1] | routes [R] | ranges1 | ranges2
__host__ __device__ inline int ws_active_off() { return 16; }
__host__ __device__ inline int ws_aoff_off(int E) { return 16 + E; }
__host__ __device__ inline int ws_routes_off(int E) { return 16 + 2 * E + 1; }
__host__ __device__ inline int ws_ranges_off(int E, int R, int which) {
    return 16 + 2 * E + 1 + R + which * (GV_MAX_GRID + 1);
}

struct WsLayout {
    size_t ints_off, info_off;
    size_t gu_off;     // float [KS][2][R][F] gate/up partial sums (KS > 1)
    size_t h_off;      // float [R][F] silu(gate) * up
    size_t first_off;  // u64 [2 launches][GV_MAX_GRID][GV_WARPS] source image of each warp's first unit
    size_t total;
};

inline WsLayout ws_layout(int T, int H, int F, int qtype, int E, int k) {
    WsLayout L;
    const size_t R = (size_t)T * k;
    GvPlan pl;
    if (!gv_plan(T, H, F, qtype, gv_n_act_max(T, E, k), &pl)) pl.KS = 1;
    const size_t ints = 16 + 2 * (size_t)E + 1 + R + 2 * (GV_MAX_GRID + 1);
    L.ints_off = 0;
    L.info_off = (ints * 4 + 255) / 256 * 256;
    L.gu_off = L.info_off + ((size_t)gv_n_virt_max(T, E, k) * sizeof(ActInfo) + 255) / 256 * 256;
    const size_t gu = pl.KS > 1 ? (size_t)pl.KS * 2 * R * F * 4 : 0;
    L.h_off = L.gu_off + (gu + 255) / 256 * 256;
    L.first_off = L.h_off + (R * F * 4 + 255) / 256 * 256;
    L.total = L.first_off + (size_t)2 * GV_MAX_GRID * GV_WARPS * 8;
    return L;
}

// how a chunk reaches its ring stage
#define GV_BULK 0  // bulk copy from the slot (HBM)
#define GV_FILL 1  // cp.async pieces from the pinned host image (a miss of a device-managed pool)
#define GV_SKIP 2  // nothing (invalid slot): the stage barrier completes without bytes

struct FfnParams {
    const void *x;
    int T, H, F, k, E, KS, RT, TPU;
    const float *weights;
    const int32_t *ws_ints;
    const int32_t *ranges;  // this launch's CTA boundaries: CTA c takes units [ranges[c], ranges[c+1])
    const ActInfo *info;
    float *gu;
    float *h;
    float *partial;
    const unsigned long long *first;  // [CTA][warp]: image of the warp's first unit, 0: none/skip/fill
    int *status;
    int sync_extra;                     // fused launch: arrivals its grid barrier waits for beyond the
                                        // grid (0; 1 only under test fault injection)
    unsigned long long sync_wait_ns;    // fused launch: bound of each grid-barrier wait
    int x_vec;              // x is 16-byte aligned: vector loads
    GvGeom geo;             // this launch's geometry
};

__device__ __forceinline__ void mbar_arrive_plain(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// Wall time in nanoseconds (the global timer).
__device__ __forceinline__ unsigned long long gv_globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bound of the drain after a timed-out wait (copies still landing in a warp's ring).
#define GV_DRAIN_NS 4000000000ull

// ------------------------------------------------------------------ fp16 fragments

// d = A B + c for one m16n8k16 tile: A 16x16 fp16 (row-major fragments), B 16x8 fp16, fp32
// accumulation.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1, const float (&c)[4]) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Two codes of a word of offset-binary bytes q + 128 (chosen by sel) as an fp16 pair of
// exact integers: the byte under an 0x64 high byte reads 1024 + (q + 128); subtracting
// 1152 leaves q.
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<const __half2 *>(&u); }
__device__ __forceinline__ uint32_t q8_pair(uint32_t t, uint32_t sel) {
    return hsub2_u(__byte_perm(t, 0x64646464u, sel), 0x64806480u);
}

// 4-bit codes of a word (nibble j = column j of its 8): nibbles 0 and 4 as an fp16 pair
// (1024 + q, minus 1024), and nibbles 1 and 5 ((1024 + 16 q) / 16 - 64).  The word shifted
// right by 8 gives nibbles 2, 6 and 3, 7 the same way.
__device__ __forceinline__ uint32_t q4_even(uint32_t w) {
    return hsub2_u((w & 0x000F000Fu) | 0x64006400u, 0x64006400u);
}
__device__ __forceinline__ uint32_t q4_odd(uint32_t w) {
    return hfma2_u((w & 0x00F000F0u) | 0x64006400u, 0x2C002C00u, 0xD400D400u);
}

// ------------------------------------------------------------------ one chunk of a unit
//
// Fragment layout.  Lane (r = lane/4, c = lane%4) holds, for the 16-row group hr of a tile,
// rows 16 hr + r and 16 hr + r + 8, and for a 32-column block the columns 8c .. 8c+7: the
// first k16 step of the block takes columns 8c+{0,1} (as k = 2c+{0,1}) and 8c+{2,3} (as
// k = 2c+8+{0,1}), the second step 8c+{4,5} and 8c+{6,7} (4-bit: the pairs (0,4), (1,5)
// and (2,6), (3,7) of the 8, which is why the staged 4-bit activations are permuted the
// same way within each group of 8).  The B fragment of a lane is then the 16 bytes of fp16
// activations at columns 8c .. 8c+7 of its B row, one shared-memory load per block.
// B rows: column n is route slot n / 2 of the virtual expert, its hi part (n even) or lo
// part (n odd).

// acc[i][hr][j]: tile i, row 16 hr + r (+ 8 for j >= 2), column 2c + (j & 1): route slot c,
// hi part (j even) or lo part.  brow: this lane's B row at the chunk's first column (plus
// 16 c bytes); as: the 4-bit block sums of route slot c's token at the chunk's first block
// (stride NTS per block), added with the block minimum to the hi columns.
template <int QT, int NTL>
__device__ __forceinline__ void chunk_dot(const unsigned char *st, int tb, int cb, const unsigned char *brow,
                                          const float *as_, int NTS, int lane, float (&acc)[NTL][2][4]) {
    constexpr int TBB = QT == MOE_Q8_0 ? 1088 : 640;  // tile block: codes, then 32 scale entries
    constexpr int SC = QT == MOE_Q8_0 ? 1024 : 512;   // offset of the scales in a tile block
    const int r = lane >> 2, c = lane & 3;
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int b = 0; b < cb; ++b) {
        const uint4 bf = *(const uint4 *)(brow + 64 * b);
        float as = 0.f;
        if constexpr (QT == MOE_Q4_SM) as = as_[b * NTS];
#pragma unroll
        for (int i = 0; i < NTL; ++i) {
            const unsigned char *blk = st + (size_t)i * tb + (size_t)b * TBB;
            // the scale entries of rows r, r+8, r+16, r+24 are adjacent (moe_scale_pos)
            float dd[4], mm[4];
            if constexpr (QT == MOE_Q8_0) {
                const uint2 e = *(const uint2 *)(blk + SC + 8 * r);
                dd[0] = __low2float(u32_as_h2(e.x)); dd[1] = __high2float(u32_as_h2(e.x));
                dd[2] = __low2float(u32_as_h2(e.y)); dd[3] = __high2float(u32_as_h2(e.y));
                mm[0] = mm[1] = mm[2] = mm[3] = 0.f;
            } else {
                const uint4 e = *(const uint4 *)(blk + SC + 16 * r);
                const uint32_t ew[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    dd[q] = __low2float(u32_as_h2(ew[q]));
                    mm[q] = __high2float(u32_as_h2(ew[q]));
                }
            }
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int R0 = 16 * hr + r;
                uint32_t A0[4], A1[4];
                if constexpr (QT == MOE_Q8_0) {  // offset-binary codes: no sign flip needed
                    // piece c / 2 (its rows rotated by 4 c / 2: see moe_piece_in_block)
                    const int pc = c >> 1;
                    const unsigned char *cp = blk + pc * 512 + (c & 1) * 8;
                    const uint2 w0 = *(const uint2 *)(cp + ((R0 + 4 * pc) & 31) * 16);
                    const uint2 w1 = *(const uint2 *)(cp + ((R0 + 8 + 4 * pc) & 31) * 16);
                    A0[0] = q8_pair(w0.x, 0x4140); A0[1] = q8_pair(w1.x, 0x4140);
                    A0[2] = q8_pair(w0.x, 0x4342); A0[3] = q8_pair(w1.x, 0x4342);
                    A1[0] = q8_pair(w0.y, 0x4140); A1[1] = q8_pair(w1.y, 0x4140);
                    A1[2] = q8_pair(w0.y, 0x4342); A1[3] = q8_pair(w1.y, 0x4342);
                } else {
                    const unsigned char *cp = blk + 4 * c;
                    const uint32_t w0 = *(const uint32_t *)(cp + R0 * 16);
                    const uint32_t w1 = *(const uint32_t *)(cp + (R0 + 8) * 16);
                    const uint32_t v0 = w0 >> 8, v1 = w1 >> 8;
                    A0[0] = q4_even(w0); A0[1] = q4_even(w1); A0[2] = q4_odd(w0); A0[3] = q4_odd(w1);
                    A1[0] = q4_even(v0); A1[1] = q4_even(v1); A1[2] = q4_odd(v0); A1[3] = q4_odd(v1);
                }
                const float d0 = dd[2 * hr], d1 = dd[2 * hr + 1], m0 = mm[2 * hr], m1 = mm[2 * hr + 1];
                float C[4];
                mma16816(C, A0[0], A0[1], A0[2], A0[3], bf.x, bf.y, zero);
                mma16816(C, A1[0], A1[1], A1[2], A1[3], bf.z, bf.w, C);
                float *a = acc[i][hr];
                a[0] = fmaf(d0, C[0], a[0]);
                a[1] = fmaf(d0, C[1], a[1]);
                a[2] = fmaf(d1, C[2], a[2]);
                a[3] = fmaf(d1, C[3], a[3]);
                if (QT == MOE_Q4_SM) {  // the block minimum times the hi column's sum
                    a[0] = fmaf(m0, as, a[0]);
                    a[2] = fmaf(m1, as, a[2]);
                }
            }
        }
    }
}

// Hi and lo parts of this lane's route slot added (columns 2c and 2c + 1: j = 0, 1 for row r,
// j = 2, 3 for row r + 8) and the route's token scale removed, into acc[i][hr][0] (row r) and
// acc[i][hr][2] (row r + 8).
template <int NTL>
__device__ __forceinline__ void finish_acc(float (&acc)[NTL][2][4], float inv) {
#pragma unroll
    for (int i = 0; i < NTL; ++i)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            acc[i][hr][0] = (acc[i][hr][0] + acc[i][hr][1]) * inv;
            acc[i][hr][2] = (acc[i][hr][2] + acc[i][hr][3]) * inv;
        }
}

// ------------------------------------------------------------------ staging the activations

// Eight consecutive activations of one source row at column col: G1 reads row `row` of x
// (a token), G2 row `row` (a route position) of h.
template <int XT, bool DOWN>
__device__ __forceinline__ void act_load8(const FfnParams &p, int row, int col, float (&v)[8]) {
    if (DOWN) {
        const size_t q = (size_t)row * p.F + col;
        const float4 a = __ldcg((const float4 *)(p.h + q)), b = __ldcg((const float4 *)(p.h + q + 4));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        const size_t off = (size_t)row * p.H + col;
        // x is read through L2: the gate/up kernel stages it before its dependency wait
        if (XT == MOE_BF16) {
            const __nv_bfloat16 *xb = (const __nv_bfloat16 *)p.x + off;
            if (p.x_vec) {
                const uint4 r = __ldcg((const uint4 *)xb);
                const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(*(const __nv_bfloat162 *)&w[e]);
                    v[2 * e] = f.x;
                    v[2 * e + 1] = f.y;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    v[e] = __bfloat162float(__ushort_as_bfloat16(__ldcg((const unsigned short *)xb + e)));
            }
        } else {
            const float *xf = (const float *)p.x + off;
            if (p.x_vec) {
                const float4 a = __ldcg((const float4 *)xf), b = __ldcg((const float4 *)(xf + 4));
                v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = __ldcg(xf + e);
            }
        }
    }
}

// One token row of a pair's slot, by one warp: the activations y = x * sc over the pair's
// K range [c0, c0 + Kr) with sc a power of two putting max |y| in [2^14, 2^15), stored as
// fp16 hi = rn(y) (row 2t) and lo = rn(y - hi) (row 2t + 1); 1/sc at inv[t]; for the 4-bit
// format the fp32 block sums of y at asum[b][t] (row stride NTS) and the columns of each
// group of 8 in the order 0 4 1 5 2 6 3 7.
template <int QT, int XT, bool DOWN, typename Mid>
__device__ void stage_row(const FfnParams &p, int row, int c0, int Kr, unsigned char *slot, int NTS, int t,
                          int lane, Mid &&mid) {
    const int RS = gv_row_stride(Kr);
    float amax = 0.f;
    float keep[2][8];  // the first 512 columns stay in registers for the second pass
#pragma unroll
    for (int i = 0; i < 2; ++i)
        if (256 * i + 8 * lane < Kr) act_load8<XT, DOWN>(p, row, c0 + 256 * i + 8 * lane, keep[i]);
    mid();  // the first loads are in flight
#pragma unroll
    for (int i = 0; i < 2; ++i)
        if (256 * i + 8 * lane < Kr)
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(keep[i][e]));
    for (int base = 512; base < Kr; base += 256) {
        const int col = base + 8 * lane;
        if (col < Kr) {
            float v[8];
            act_load8<XT, DOWN>(p, row, c0 + col, v);
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int ex = amax > 0.f ? ((__float_as_int(amax) >> 23) & 0xFF) - 127 : 0;
    ex = max(ex, -100);  // subnormal maxima: any scale keeps them exact enough
    const float sc = __int_as_float((127 + 14 - ex) << 23);
    float *inv = (float *)(slot + GV_INV_OFF(NTS, RS));
    float *asum = (float *)(slot + GV_ASUM_OFF(NTS, RS));
    if (lane == 0) inv[t] = __int_as_float((127 - 14 + ex) << 23);
    __half *hi = (__half *)(slot + (size_t)(2 * t) * RS);
    __half *lo = (__half *)(slot + (size_t)(2 * t + 1) * RS + GV_LO_SHIFT);
    // one step of 8 columns per lane; every lane calls it (the 4-bit block sums shuffle)
    auto emit = [&](int col, const float (&v)[8]) {
        float bs = 0.f;
        if (col < Kr) {
            __align__(16) __half h8[8];
            __align__(16) __half l8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float y = v[e] * sc;
                const __half hh = __float2half_rn(y);
                const __half ll = __float2half_rn(y - __half2float(hh));
                const int at = QT == MOE_Q4_SM ? ((e & 3) * 2 + (e >> 2)) : e;
                h8[at] = hh;
                l8[at] = ll;
                bs += y;
            }
            *(uint4 *)(hi + col) = *(const uint4 *)h8;
            *(uint4 *)(lo + col) = *(const uint4 *)l8;
        }
        if (QT == MOE_Q4_SM) {  // 4 lanes cover one 32-column block
            bs += __shfl_xor_sync(0xffffffffu, bs, 1);
            bs += __shfl_xor_sync(0xffffffffu, bs, 2);
            if (col < Kr && (lane & 3) == 0) asum[(col / 32) * NTS + t] = bs;
        }
    };
#pragma unroll
    for (int i = 0; i < 2; ++i)
        if (256 * i < Kr) emit(256 * i + 8 * lane, keep[i]);
    for (int base = 512; base < Kr; base += 256) {
        const int col = base + 8 * lane;
        float v[8] = {};
        if (col < Kr) act_load8<XT, DOWN>(p, row, c0 + col, v);
        emit(col, v);
    }
}

// ------------------------------------------------------------------ fills

// Issues one fill chunk into a ring stage (whole warp): the runs of n16 16-byte pieces of its
// tiles (src0 for tile 0, src1 for tile NTL - 1; at most two tiles) as cp.async pieces tied to
// the stage barrier, then lane 0's arrival.  Kept out of line: the resident path stays free of
// its registers.
__device__ __noinline__ void issue_fill(uint64_t *bar, unsigned char *dst, const uint8_t *src0,
                                        const uint8_t *src1, int ntl, int tb, int n16, int lane) {
    for (int i = 0; i < ntl; ++i) {
        const uint8_t *src = (i ? src1 : src0) + 16 * lane;
        unsigned char *d = dst + (size_t)i * tb + 16 * lane;
        for (int j = lane; j < n16; j += 32, src += 512, d += 512) cp_async_16(d, src);
    }
    cp_async_mbar_arrive(bar);
    __syncwarp();  // every lane's pieces are counted before lane 0's arrival
    if (lane == 0) mbar_arrive_plain(bar);
}

// A chunk of a unit whose expert missed arrives in its ring stage from the expert's pinned
// host image over the CPU-GPU link (cp.async pieces, issued S stages ahead like the bulk
// copies of resident chunks).  The first virtual expert of the expert also writes the chunk's
// bytes (one run of tile blocks per tile) from the stage to the same offsets of the expert's
// slot, so the slot holds the image once every chunk has passed.
template <int QT>
__device__ void write_through(const ActInfo &in, int H, int F, bool down, int NTL, int g, int kb0, int cb,
                              const unsigned char *st, int tb, int lane) {
    const int K = down ? F : H;
    const int n16 = cb * moe_tile_block_bytes(QT) / 16;
    for (int i = 0; i < NTL; ++i) {
        const size_t off = moe_expert_matrix_offset(QT, H, F, down ? 2 : i) +
                           moe_tile_block_offset(QT, K, down ? g + i : g, kb0);
        uint4 *dst = (uint4 *)((uint8_t *)in.dst + off);
        const uint4 *tile = (const uint4 *)(st + (size_t)i * tb);
        for (int j = lane; j < n16; j += 32) __stcs(dst + j, tile[j]);
    }
}

// ------------------------------------------------------------------ R1: K-split reduction

// h[q] = silu(sum gate) * (sum up) over the K-split partial sums gu [KS][2][R][F], the K
// ranges summed in order, for every route position q of the call (n = R * F elements, one per
// thread, all partials of a thread in flight).  Runs between the gate/up and the down GEMV
// when the gate/up kernel split K.
template <int KS>
__device__ __forceinline__ void ks_reduce_range(const float *__restrict__ gu, float *__restrict__ h, size_t n,
                                                size_t q0, size_t step) {
    for (size_t q = q0; q < n; q += step) {
        float gp[KS], up[KS];
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            gp[k] = __ldcg(gu + (size_t)(2 * k) * n + q);
            up[k] = __ldcg(gu + (size_t)(2 * k + 1) * n + q);
        }
        float gs = 0.f, us = 0.f;
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            gs += gp[k];
            us += up[k];
        }
        h[q] = silu_mul(gs, us);
    }
}

template <int KS>
__global__ void __launch_bounds__(256) ks_reduce_kernel(const float *__restrict__ gu, float *__restrict__ h,
                                                        size_t n) {
    pdl_wait();
    pdl_trigger();
    ks_reduce_range<KS>(gu, h, n, (size_t)blockIdx.x * 256 + threadIdx.x, (size_t)gridDim.x * 256);
}

// ------------------------------------------------------------------ G1 / G2: the warp-ring kernel
//
// Units of a virtual expert: G1 has KS K ranges x F/32 row tiles, ordered (ks, g); unit
// (ks, g) holds the gate and the up tile g over K range ks.  G2 has H/(32 NTL) groups of
// NTL down tiles over the whole of F.  A pair = (virtual expert, K range) shares one staged
// activation slot; a CTA stages the pairs of its unit range in phases of at most
// act_slots pairs (usually one phase), between CTA barriers.
//
// Warp ring: the warp's chunks (its units in turn within each phase, each unit cut into
// chunks of CB blocks) go through S stages; chunk J lives in stage J % S and completes phase
// (J / S) & 1 of that stage's mbarrier, on which every lane waits.  Lane 0 issues chunk J+S
// into the stage once all lanes are done with chunk J (after a __syncwarp).  A fill chunk or
// a skipped expert's chunk arrives on its mbarrier without bytes.

// The stage barriers of warp `warp` for the gate/up (DOWN false) or the down GEMV.
template <bool DOWN>
__device__ __forceinline__ uint64_t *gv_bars(unsigned char *smem, int warp) {
    return (uint64_t *)smem + (DOWN ? GV_WARPS * GV_MAX_STAGES : 0) + warp * GV_MAX_STAGES;
}

// One GEMV over this CTA's unit range.  `gate()` is called once by every thread of the CTA
// before anything produced by the earlier stages of the call (activations, h) is read:
// at once when PRIME is false; when PRIME is true, after each warp's lane 0 has issued the
// weight copies of its whole ring (they depend only on the routing metadata).
template <int QT, int XT, bool DOWN, int NTL, bool PRIME, typename Gate>
__device__ __forceinline__ void ffn_body(const FfnParams &p, unsigned char *smem, Gate &&gate) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *bars = gv_bars<DOWN>(smem, warp);
    const int u0 = p.ranges[blockIdx.x], u1 = p.ranges[blockIdx.x + 1];
    const unsigned long long first_src = !PRIME && lane == 0 ? p.first[blockIdx.x * GV_WARPS + warp] : 0ull;
    if (u0 >= u1) {
        gate();
        return;
    }
    constexpr int TBB = QT == MOE_Q8_0 ? 1088 : 640;  // bytes of a tile block (codes + scales)
    const GvGeom G = p.geo;
    const int K = DOWN ? p.F : p.H;
    const int nbr = G.nbr, Kr = nbr * 32, CB = G.CB;
    const int upp = DOWN ? (p.H / 32) / NTL : p.F / 32;  // units per pair
    const int tb = CB * TBB;                              // tile stride in a stage
    const int nch = (nbr + CB - 1) / CB;                  // chunks per unit
    const int RS = gv_row_stride(Kr);
    const int NTS = DOWN ? GV_TOK : p.T;  // token rows of a slot
    const int n_w = min(GV_WARPS, u1 - u0);
    const int S = min(GV_MAX_STAGES, G.ring_bytes / (n_w * G.chunk_bytes));
    unsigned char *ring = smem + GV_BARS + (size_t)warp * S * G.chunk_bytes;
    unsigned char *act_region = smem + GV_BARS + G.ring_bytes;

    // Pairs are ordered (K range, virtual expert) in the gate/up launch — CTA c works on K range
    // c / (G / KS) only, so it stages x before its dependency wait — and by virtual expert in
    // the down launch.
    const int nv = DOWN ? 1 : __ldcg(p.ws_ints + 1);  // virtual experts of the call
    auto pair_v = [&](int pair) { return DOWN ? pair : pair % nv; };
    auto decode = [&](int u, int &v, int &pair, int &ks, int &g) {
        pair = u / upp;
        ks = DOWN ? 0 : pair / nv;
        v = DOWN ? pair : pair - ks * nv;
        g = (u - pair * upp) * (DOWN ? NTL : 1);
    };
    // a phase covers the units of act_slots consecutive pairs (slot = pair - first pair)
    auto phase_end = [&](int a) { return min(u1, (a / upp + G.act_slots) * upp); };

    // ---- producer state (the same in every lane): the next chunk to issue
    int pc_ph1 = u0, pc_u = u1, pc_ch = 0;  // phase end, unit (u1: none left), chunk
    int pc_cached_v = -1;
    unsigned long long pc_src = 0ull;
    int pc_kind = GV_SKIP;
    auto pc_info = [&]() {  // where the weights of the next chunk's virtual expert are read from
        const int v = pair_v(pc_u / upp);
        if (v != pc_cached_v) {
            const ActInfo &in = p.info[v];
            pc_src = in.src;
            pc_kind = in.n_e == 0 ? GV_SKIP : in.fill ? GV_FILL : GV_BULK;
            pc_cached_v = v;
        }
    };
    auto pc_first = [&](int a) {  // this warp's first unit at or after phase start a
        pc_u = u1;
        while (a < u1) {
            const int e = phase_end(a);
            if (a + warp < e) {
                pc_ph1 = e;
                pc_u = a + warp;
                pc_ch = 0;
                return;
            }
            a = e;
        }
    };
    auto pc_next = [&]() {
        if (++pc_ch < nch) return;
        pc_ch = 0;
        pc_u += GV_WARPS;
        if (pc_u >= pc_ph1) pc_first(pc_ph1);
    };
    // Called by the whole warp.  A resident chunk: lane 0 issues one bulk copy per tile (TMA
    // engine), counted in bytes on the stage barrier.  A fill chunk (the expert's pinned host
    // image): every lane copies its 16-byte pieces with cp.async and ties them to the stage
    // barrier, then lane 0 arrives, so the stage completes when the pieces have landed — fill
    // chunks are in flight S stages ahead like resident ones.  A skipped expert's chunk: lane 0
    // arrives without bytes.
    auto issue = [&](int stage) {
        uint64_t *bar = &bars[stage];
        int v, pair, ks, g;
        decode(pc_u, v, pair, ks, g);
        pc_info();
        if (pc_kind == GV_SKIP) {
            if (lane == 0) mbar_arrive_plain(bar);
            return;
        }
        const int kb0 = ks * nbr + pc_ch * CB, cb = min(CB, nbr - pc_ch * CB);
        unsigned char *dst = ring + (size_t)stage * G.chunk_bytes;
        if (pc_kind == GV_BULK) {
            if (lane == 0) {
                mbar_arrive_expect_tx(bar, (uint32_t)(NTL * cb * TBB));
                for (int i = 0; i < NTL; ++i) {
                    const uint8_t *mat =
                        (const uint8_t *)pc_src + moe_expert_matrix_offset(QT, p.H, p.F, DOWN ? 2 : i);
                    bulk_g2s(dst + (size_t)i * tb, mat + moe_tile_block_offset(QT, K, DOWN ? g + i : g, kb0),
                             (uint32_t)(cb * TBB), bar);
                }
            }
            return;
        }
        const uint8_t *img = (const uint8_t *)pc_src;
        issue_fill(bar, dst, img + moe_expert_matrix_offset(QT, p.H, p.F, DOWN ? 2 : 0) +
                                 moe_tile_block_offset(QT, K, g, kb0),
                   img + moe_expert_matrix_offset(QT, p.H, p.F, DOWN ? 2 : NTL - 1) +
                       moe_tile_block_offset(QT, K, DOWN ? g + NTL - 1 : g, kb0),
                   NTL, tb, cb * TBB / 16, lane);
    };

    int J_issued = 0;    // chunks issued by this warp
    bool dead = false;   // a wait ran out: no more waits, copies or outputs
    // issue chunks until `limit` have been issued (chunk X goes to stage X % S, which chunk
    // X - S has left); warp-uniform
    auto top_up = [&](int limit) {
        if (dead) return;
        while (J_issued < limit && pc_u < u1) {
            issue(J_issued % S);
            pc_next();
            ++J_issued;
        }
    };
    pc_first(u0);
    if (PRIME) {
        top_up(S);
    } else {
        const unsigned long long fs = __shfl_sync(0xffffffffu, first_src, 0);
        if (pc_u == u0 + warp && fs) {  // the permute kernel resolved it: issue at once
            pc_src = fs;
            pc_kind = GV_BULK;
            pc_cached_v = pair_v(pc_u / upp);
            top_up(1);
        } else if (pc_u < u1) {
            pc_info();
        }
    }
    __syncwarp();
    gate();

    int J = 0;           // chunks this warp has reached
    int J_done = 0;      // chunks whose stage completed (waited on)
    for (int a = u0; a < u1;) {
        const int e = phase_end(a);
        const int pr0 = a / upp, npr = (e - 1) / upp - pr0 + 1;
        if (a != u0) __syncthreads();  // the previous phase's slots are no longer read
        // Staging, item (pair i, token row t).  Gate/up: every token of the call over the
        // pair's K range, read from x without the routing metadata.  Down: the routes of the
        // pair's virtual expert, read from h.  Row 0's item also writes the slot header.
        // the warp's first chunk goes out once its first staging loads are in flight (or at
        // once for a warp without staging work), ahead of the conversion; the rest of its ring
        // is filled at its first wait, so that every warp's first chunk is ahead of them in the
        // copy engine's queue
        auto first_issue = [&]() {
            if (a == u0) top_up(1);
        };
        if (!DOWN) {  // x is staged (slot 0's rows); each pair's slot holds its header
            if (a == u0) top_up(S);
            for (int i = warp; i < npr; i += GV_WARPS)
                if (lane == 0)
                    ((SlotHdr *)(act_region + (size_t)i * G.slot_bytes + GV_HDR_OFF(NTS, RS)))->in =
                        p.info[pair_v(pr0 + i)];
        }
        for (int it = warp; DOWN && it < npr * NTS; it += GV_WARPS) {
            const int i = it / NTS, t = it - i * NTS;
            const int v = pr0 + i;
            unsigned char *slot = act_region + (size_t)i * G.slot_bytes;
            SlotHdr *hdr = (SlotHdr *)(slot + GV_HDR_OFF(NTS, RS));
            {
                const ActInfo in = p.info[v];
                if (t == 0 && lane == 0) hdr->in = in;
                if (t < in.n_e) {
                    if (lane == 0) hdr->w[t] = p.weights[in.rt[t]];
                    stage_row<QT, XT, DOWN>(p, in.pos0 + t, 0, Kr, slot, NTS, t, lane, first_issue);
                } else if (QT == MOE_Q4_SM) {
                    float *asum = (float *)(slot + GV_ASUM_OFF(NTS, RS));
                    for (int b = lane; b < nbr; b += 32) asum[b * NTS + t] = 0.f;
                }
            }
        }
        first_issue();
        __syncthreads();

        for (int u = a + warp; u < e; u += GV_WARPS) {
            int v, pair, ks, g;
            decode(u, v, pair, ks, g);
            const unsigned char *hslot = act_region + (size_t)(pair - pr0) * G.slot_bytes;
            const SlotHdr *hdr = (const SlotHdr *)(hslot + GV_HDR_OFF(NTS, RS));
            const unsigned char *slot = DOWN ? hslot : act_region;  // the staged activations
            const int n_e = hdr->in.n_e, fill = hdr->in.fill;
            // Token row of route slot q of this virtual expert in the staged slot (gate/up: the
            // route's token; down: q); slots past n_e read row 0 (their columns are not used).
            auto trow = [&](int q) { return q >= n_e ? 0 : (DOWN ? q : hdr->in.rt[q] / p.k); };
            const int r_ = lane >> 2, c_ = lane & 3;
            // B row of column r_: route slot r_ / 2, hi (r_ even) or lo (64 bytes into its row)
            const unsigned char *brow =
                slot + (size_t)(2 * trow(r_ >> 1) + (r_ & 1)) * RS + (r_ & 1) * GV_LO_SHIFT + 16 * c_;
            // the lane's two accumulator columns 2c, 2c+1: route slot c, hi and lo
            const int trc = trow(c_);
            const float *asb = (const float *)(slot + GV_ASUM_OFF(NTS, RS));
            float acc[NTL][2][4];
#pragma unroll
            for (int i = 0; i < NTL; ++i)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][hr][j] = 0.f;
            for (int ch = 0; ch < nch; ++ch, ++J) {
                const int stg = J % S;
                unsigned char *st = ring + (size_t)stg * G.chunk_bytes;
                top_up(J + S);
                if (!dead) {
                    const bool ok = mbar_wait_bounded(&bars[stg], (J / S) & 1, p.status);
                    if (__all_sync(0xffffffffu, ok)) J_done = J + 1;
                    else dead = true;
                }
                if (!dead && n_e > 0) {
                    const int cb = min(CB, nbr - ch * CB);
                    if (fill && hdr->in.wt)  // the first group of a missed expert fills its slot
                        write_through<QT>(hdr->in, p.H, p.F, DOWN, NTL, g, ks * nbr + ch * CB, cb, st, tb, lane);
                    chunk_dot<QT, NTL>(st, tb, cb, brow + (size_t)64 * ch * CB, asb + (size_t)ch * CB * NTS + trc, NTS,
                                       lane, acc);
                    // the stage was written through the generic proxy (cp.async); a later bulk
                    // copy (async proxy) overwrites it
                    if (fill) fence_proxy_async_smem();
                }
                __syncwarp();  // every lane is done with the stage
                top_up(J + 1 + S);
            }
            if (dead || n_e == 0) continue;
            const float *inv = (const float *)(slot + GV_INV_OFF(NTS, RS));
            finish_acc<NTL>(acc, inv[trc]);
            const int r = lane >> 2, c = lane & 3, pos0 = hdr->in.pos0;
            const int t = c;  // this lane's route slot
#pragma unroll
            for (int j = 0; j < 4; j += 2) {
                if (t >= n_e) continue;
                const int pos = pos0 + t;
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int row = 16 * hr + r + 8 * (j >> 1);
                    if (DOWN) {
                        const int rt = hdr->in.rt[t];
                        const float w = hdr->w[t];
#pragma unroll
                        for (int i = 0; i < NTL; ++i)
                            p.partial[(size_t)rt * p.H + 32 * (g + i) + row] = w * acc[i][hr][j];
                    } else if (p.KS == 1) {
                        p.h[(size_t)pos * p.F + 32 * g + row] = silu_mul(acc[0][hr][j], acc[NTL - 1][hr][j]);
                    } else {
                        p.gu[(((size_t)ks * 2 + 0) * p.RT + pos) * p.F + 32 * g + row] = acc[0][hr][j];
                        p.gu[(((size_t)ks * 2 + 1) * p.RT + pos) * p.F + 32 * g + row] = acc[NTL - 1][hr][j];
                    }
                }
            }
        }
        a = e;
    }
    // Never leave with copies in flight: a wait that ran out left chunks J_done .. issued-1
    // unconsumed.  Keep waiting for each (the status word already says MOE_ERR_TIMEOUT), up to
    // GV_DRAIN_NS of wall time in all, so that the CTA exits only after its copies landed
    // unless the copy engine itself stopped answering.
    if (lane == 0 && J_done < J_issued) {
        const unsigned long long t0 = gv_globaltimer();
        for (int j = J_done; j < J_issued; ++j)
            while (!mbar_try_wait(&bars[j % S], (j / S) & 1))
                if (gv_globaltimer() - t0 > GV_DRAIN_NS) return;
    }
}

// Gate/up launch: CTA c works on K range c / (G / KS) only, so it stages x (every token row
// over that range, into slot 0) before its dependency wait.  x is complete when the grid
// starts: the launch is ordered behind the call's permute kernel, which lets the next grid
// start only once everything before it has completed (or behind a full completion).
template <int QT, int XT>
__device__ __forceinline__ void stage_x_static(const FfnParams &p, unsigned char *smem) {
    const GvGeom G = p.geo;
    const int Kr = G.nbr * 32, ks = blockIdx.x / (gridDim.x / p.KS);
    unsigned char *slot0 = smem + GV_BARS + G.ring_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (ks >= p.KS) return;
    for (int t = warp; t < p.T; t += GV_WARPS) stage_row<QT, XT, false>(p, t, ks * Kr, Kr, slot0, p.T, t, lane, [] {});
}

template <int QT, int XT, bool DOWN, int NTL>
__global__ void __launch_bounds__(GV_THREADS, 1) ffn_warp_kernel(FfnParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    if ((threadIdx.x & 31) == 0) {  // before the dependency wait: every stage barrier this warp may use
        uint64_t *bars = gv_bars<DOWN>(smem, threadIdx.x >> 5);
        for (int s = 0; s < GV_MAX_STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    if (!DOWN) stage_x_static<QT, XT>(p, smem);
    pdl_wait();  // ranges, routing (and h) come from earlier kernels
    pdl_trigger();
    ffn_body<QT, XT, DOWN, NTL, false>(p, smem, [] {});
}

// ------------------------------------------------------------------ G1 + R1 + G2 in one launch
//
// All CTAs are resident at once (cooperative launch, grid within the occupancy).  Each CTA
// runs its gate/up units, then issues the weight copies of its down units into its rings
// (the down weights depend only on the routing), and only then waits at a grid barrier for
// every CTA's gate/up results; with a K split the grid forms h between two barriers.  The
// down kernel's ramp-up thus overlaps the gate/up kernel's tail instead of following it.

// Grid barrier: sync[0] counts the CTAs that arrived, sync[1] is the barrier's generation.
// The last CTA to arrive resets the count and advances the generation, so the barrier can be
// passed any number of times (sync[0] starts at 0: the permute kernel clears it).  The wait
// is bounded: past wait_ns (GV_GRID_WAIT_NS normally) the CTA sets MOE_ERR_TIMEOUT and goes
// on.  `extra` raises the arrival count the barrier waits for above the grid size; it is 0
// except under test fault injection, where 1 makes every CTA's wait run out.
#define GV_GRID_WAIT_NS 500000000ull
#define GV_GRID_WAIT_TEST_NS 20000000ull
__device__ __forceinline__ int ld_acquire_gpu(const int *a) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}
__device__ void grid_sync(int *sync, int *status, int extra, unsigned long long wait_ns) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const int gen = ld_acquire_gpu(sync + 1);
        __threadfence();  // this CTA's writes before its arrival
        if (atomicAdd(sync, 1) == (int)gridDim.x + extra - 1) {
            atomicExch(sync, 0);
            __threadfence();
            atomicAdd(sync + 1, 1);
        } else {
            const unsigned long long t0 = gv_globaltimer();
            while (ld_acquire_gpu(sync + 1) == gen) {
                if (gv_globaltimer() - t0 > wait_ns) {
                    moe_set_status(status, MOE_ERR_TIMEOUT);
                    break;
                }
                __nanosleep(32);
            }
        }
        __threadfence();
    }
    __syncthreads();
}

template <int QT, int XT, int NTL2>
__global__ void __launch_bounds__(GV_THREADS, 1) ffn_fused_kernel(FfnParams p1, FfnParams p2, int *sync) {
    extern __shared__ __align__(128) unsigned char smem[];
    if ((threadIdx.x & 31) == 0) {
        uint64_t *b1 = gv_bars<false>(smem, threadIdx.x >> 5), *b2 = gv_bars<true>(smem, threadIdx.x >> 5);
        for (int s = 0; s < GV_MAX_STAGES; ++s) {
            mbar_init(&b1[s], 1);
            mbar_init(&b2[s], 1);
        }
        fence_mbar_init();
    }
    stage_x_static<QT, XT>(p1, smem);
    pdl_wait();
    pdl_trigger();
    ffn_body<QT, XT, false, 2, false>(p1, smem, [] {});
    __syncthreads();  // the gate/up rings and slots are no longer read: the down rings reuse them
    ffn_body<QT, MOE_F32, true, NTL2, true>(p2, smem, [&] {
        grid_sync(sync, p1.status, p1.sync_extra, p1.sync_wait_ns);
        if (p1.KS > 1) {
            const size_t n = (size_t)p1.RT * p1.F, i0 = (size_t)blockIdx.x * GV_THREADS + threadIdx.x,
                         step = (size_t)gridDim.x * GV_THREADS;
            switch (p1.KS) {
                case 2: ks_reduce_range<2>(p1.gu, p2.h, n, i0, step); break;
                case 4: ks_reduce_range<4>(p1.gu, p2.h, n, i0, step); break;
                case 8: ks_reduce_range<8>(p1.gu, p2.h, n, i0, step); break;
                default: ks_reduce_range<16>(p1.gu, p2.h, n, i0, step); break;
            }
            grid_sync(sync, p1.status, p1.sync_extra, p1.sync_wait_ns);
        }
    });
}

// ------------------------------------------------------------------ P1: permute

// Exclusive prefix sum over the 256 threads of the block of a 64-bit value (warp shuffles,
// then the 8 warp totals); *total receives the sum over the block.  Every thread calls it.
__device__ __forceinline__ unsigned long long block_scan_excl(unsigned long long v, unsigned long long *wsum,
                                                              unsigned long long *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    unsigned long long before = 0ull, all = 0ull;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        before += w < warp ? wsum[w] : 0ull;
        all += wsum[w];
    }
    *total = all;
    return before + x - v;
}

// Stable counting sort of the routes r = t*k + j by expert (restricted to a subset), the
// ascending list of active experts and their route ranges, the virtual experts (groups of
// at most GV_TOK routes of one expert) with where their weights are read from (slot in the
// pool, or the pinned host image for a fill, written through by the first group only), and
// the unit ranges of the CTAs of both GEMV launches.  Every unit weighs the same (its bytes,
// dequantisation and MMAs do not depend on its routes: the MMA computes every column of a
// virtual expert), so CTA c of G takes units [floor(c U / G), floor((c+1) U / G)) of the down
// launch.  The gate/up launch orders its pairs (K range, virtual expert) and gives each K
// range G1 / KS1 CTAs (G1 is a multiple of KS1): CTA c takes, within K range k = c / (G1/KS1),
// units k U' + [floor(c' U' / Gk), floor((c'+1) U' / Gk)) with U' the units of one K range,
// Gk = G1 / KS1 and c' = c - k Gk.
//
// One CTA of 256 threads, everything in shared memory, no serial loop: a route's rank among
// the earlier routes of its expert comes from a warp match (rank within the warp) plus the
// counts of the earlier warps; offsets, active-expert indices and virtual-expert bases come
// from one block-wide scan over the experts.
__global__ void __launch_bounds__(256) permute_kernel(const int32_t *__restrict__ ids, int R, int E,
                                                      const int32_t *__restrict__ subset, int n_subset,
                                                      int32_t *__restrict__ ints, ActInfo *__restrict__ info,
                                                      const int32_t *__restrict__ slot_table, int n_slots,
                                                      const uint8_t *pool, size_t slot_bytes,
                                                      const unsigned long long *__restrict__ fill_src,
                                                      int G1, int per_v1, int KS1, int G2, int per_v2,
                                                      unsigned long long *__restrict__ first, int *status) {
    static_assert(GV_PERMUTE_MAX_R <= 256 && MOE_MAX_E <= 256, "one route and one expert per thread");
    constexpr int NW = 8;  // warps
    __shared__ int cntw[NW][MOE_MAX_E];  // routes of expert e in warp w; then the earlier warps' count
    __shared__ int s_off[MOE_MAX_E], s_slot[MOE_MAX_E];
    __shared__ int s_active[MOE_MAX_E], s_aoff[MOE_MAX_E + 1], vb[MOE_MAX_E + 1];
    __shared__ unsigned long long s_fill[MOE_MAX_E], wsum[NW];
    __shared__ unsigned char insub[MOE_MAX_E];
    __shared__ int s_routes[GV_PERMUTE_MAX_R];
    __shared__ int s_rng[2][GV_MAX_GRID + 1];
    // per virtual expert: where its weights are read from (0: skip or fill), for the first-unit
    // table; up to GV_VSRC entries (the most a decode call has), the rest read back from info
    constexpr int GV_VSRC = 512;
    __shared__ unsigned long long vsrc[GV_VSRC];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();  // ids and the slot table come from earlier kernels
    pdl_trigger();
    // ---- loads (one round trip) and clears
    const int e_r = tid < R ? ids[tid] : -1;  // this thread's route
    if (tid < E) {
        s_slot[tid] = slot_table ? slot_table[tid] : tid;
        s_fill[tid] = fill_src ? fill_src[tid] : 0ull;
        insub[tid] = subset ? 0 : 1;
#pragma unroll
        for (int w = 0; w < NW; ++w) cntw[w][tid] = 0;
    }
    __syncthreads();
    if (subset) {
        for (int i = tid; i < n_subset; i += 256) {
            const int e = subset[i];
            if (e >= 0 && e < E) insub[e] = 1;
            else moe_set_status(status, MOE_ERR_INVALID);
        }
        __syncthreads();
    }
    // ---- per warp: rank of each route among the warp's routes of its expert, and counts
    int e = -1;
    if (tid < R) {  // id -1: a route dropped by the load threshold (no route, not an error)
        if (e_r < -1 || e_r >= E) moe_set_status(status, MOE_ERR_INVALID);
        else if (e_r >= 0 && insub[e_r]) e = e_r;
    }
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    const int wrank = __popc(grp & ((1u << lane) - 1u));
    if (e >= 0 && wrank == 0) cntw[warp][e] = __popc(grp);
    __syncthreads();
    // ---- per expert: count, earlier-warp counts, then the scan over experts
    int cnt = 0;
    if (tid < E) {
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const int c = cntw[w][tid];
            cntw[w][tid] = cnt;
            cnt += c;
        }
    }
    const int nvirt = (cnt + GV_TOK - 1) / GV_TOK;
    // packed (route offset, active index, virtual base): each field < 2^20
    const unsigned long long packed = (unsigned long long)cnt | ((unsigned long long)(cnt > 0) << 20) |
                                      ((unsigned long long)nvirt << 40);
    unsigned long long tot;
    const unsigned long long ex = block_scan_excl(packed, wsum, &tot);
    const int off_e = (int)(ex & 0xFFFFF), aidx = (int)((ex >> 20) & 0xFFFFF), vbase = (int)(ex >> 40);
    const int n_act = (int)((tot >> 20) & 0xFFFFF), n_routes = (int)(tot & 0xFFFFF), n_virt = (int)(tot >> 40);
    if (tid < E) {
        s_off[tid] = off_e;
        if (cnt > 0) {
            s_active[aidx] = tid;
            s_aoff[aidx] = off_e;
            vb[aidx] = vbase;
        }
    }
    if (tid == 0) {
        s_aoff[n_act] = n_routes;
        vb[n_act] = n_virt;
        ints[0] = n_act;
        ints[1] = n_virt;
        ints[GV_SYNC_OFF] = 0;  // the fused GEMV's grid barrier count
    }
    __syncthreads();
    // ---- routes in expert order (stable: warp order, then lane order)
    int *routes = ints + ws_routes_off(E);
    if (e >= 0) {
        const int pos = s_off[e] + cntw[warp][e] + wrank;
        s_routes[pos] = tid;
        routes[pos] = tid;
    }
    {
        int *active = ints + ws_active_off(), *aoff = ints + ws_aoff_off(E);
        if (tid < n_act) active[tid] = s_active[tid];
        if (tid <= n_act) aoff[tid] = s_aoff[tid];
    }
    __syncthreads();
    // ---- virtual experts of each active expert
    if (tid < n_act) {
        const int a = tid, ex_id = s_active[a], slot = s_slot[ex_id];
        const int n_e = s_aoff[a + 1] - s_aoff[a];
        ActInfo in;
        in.fill = in.wt = 0;
        in.src = in.dst = 0ull;
        // a fill source without a slot: read the host image only (an expert the pool's
        // admission policy bypassed); a slot out of range otherwise is an error
        const unsigned long long f = s_fill[ex_id];
        const bool bypass = f != 0ull && slot < 0;
        const bool bad = !bypass && (slot < 0 || slot >= n_slots);
        if (bad) {
            moe_set_status(status, MOE_ERR_INVALID);  // nothing of this expert is read
        } else {
            in.dst = bypass ? 0ull : (unsigned long long)(pool + (size_t)slot * slot_bytes);
            in.fill = f != 0ull;
            in.src = f ? f : in.dst;
        }
        for (int j = 0; j < vb[a + 1] - vb[a]; ++j) {
            in.pos0 = s_aoff[a] + GV_TOK * j;
            in.n_e = bad ? 0 : min(GV_TOK, n_e - GV_TOK * j);
            in.wt = in.fill && !bypass && j == 0;
#pragma unroll
            for (int t = 0; t < GV_TOK; ++t) in.rt[t] = t < in.n_e ? s_routes[in.pos0 + t] : 0;
            info[vb[a] + j] = in;
            if (vb[a] + j < GV_VSRC) vsrc[vb[a] + j] = in.n_e > 0 && !in.fill ? in.src : 0ull;
        }
    }
    // ---- unit ranges of both launches
    {
        int *rg1 = ints + ws_ranges_off(E, R, 0), *rg2 = ints + ws_ranges_off(E, R, 1);
        const int Gk = G1 / KS1;
        const unsigned long long Uk = (unsigned long long)n_virt * (per_v1 / KS1);
        for (int c = tid; c <= G1; c += 256) {
            const int k = c / Gk, cl = c - k * Gk;
            const int u = (int)(k * Uk + Uk * (unsigned long long)cl / (unsigned long long)Gk);
            s_rng[0][c] = u;
            rg1[c] = u;
        }
        const unsigned long long U2 = (unsigned long long)n_virt * per_v2;
        for (int c = tid; c <= G2; c += 256) {
            const int u = (int)(U2 * (unsigned long long)c / (unsigned long long)G2);
            s_rng[1][c] = u;
            rg2[c] = u;
        }
    }
    __syncthreads();
    // ---- where each warp's first unit (unit ranges[c] + warp) is read from, so that a GEMV warp
    // can issue its first copy with the range load (0: no such unit, a skip or a fill).  A
    // unit's pair is u / upp (upp units per pair); its virtual expert is the pair (down) or the
    // pair modulo n_virt (gate/up: pairs ordered (K range, virtual expert)).
#pragma unroll
    for (int l = 0; l < 2; ++l) {
        const int G = l ? G2 : G1, upp = l ? per_v2 : per_v1 / KS1;
        unsigned long long *fo = first + (size_t)l * GV_MAX_GRID * GV_WARPS;
        for (int c = tid; c < G; c += 256) {
            const int u0 = s_rng[l][c], u1 = s_rng[l][c + 1];
            const int pair = u0 / upp;
            int v = l ? pair : (n_virt ? pair % n_virt : 0), r = u0 - pair * upp;
            for (int w = 0; w < GV_WARPS; ++w) {
                unsigned long long d = 0ull;
                if (u0 + w < u1) {
                    if (v < GV_VSRC) {
                        d = vsrc[v];
                    } else {
                        const ActInfo &in = info[v];  // written above by this CTA
                        if (in.n_e > 0 && !in.fill) d = in.src;
                    }
                }
                fo[(size_t)c * GV_WARPS + w] = d;
                if (++r == upp) {
                    r = 0;
                    if (++v == n_virt && !l) v = 0;
                }
            }
        }
    }
}

// ------------------------------------------------------------------ C1: combine

__global__ void combine_kernel(const float4 *__restrict__ partial, int T, int k, int H4,
                               const float4 *extra, float4 *y) {
    const size_t n = (size_t)T * H4;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t t = i / H4, h = i % H4;
        float4 s = extra ? extra[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        // every route's load issued first, then the sum in route order
        float4 v[MOE_MAX_K];
#pragma unroll
        for (int j = 0; j < MOE_MAX_K; ++j)
            if (j < k) v[j] = partial[(t * k + j) * H4 + h];
#pragma unroll
        for (int j = 0; j < MOE_MAX_K; ++j)
            if (j < k) {
                s.x += v[j].x; s.y += v[j].y; s.z += v[j].z; s.w += v[j].w;
            }
        y[i] = s;
    }
}

// Combine + RMSNorm for the stack: one CTA per token.  y = extra + sum_j partial[j] (fixed
// order), then xn = y / sqrt(mean(y^2) + eps) with a fixed-order block reduction.
__global__ void __launch_bounds__(256) combine_norm_kernel(const float4 *__restrict__ partial, int k, int H4,
                                                           const float4 *extra, float4 *y, float4 *xn,
                                                           float eps, const int32_t *__restrict__ ids) {
    __shared__ float red[8];
    constexpr int KEEP = 4;  // sums kept in registers for the scaling pass (H <= 4096 at 256 threads)
    const int t = blockIdx.x;
    pdl_wait();  // the partial outputs come from the down GEMV
    pdl_trigger();
    float ss = 0.f;
    float4 keep[KEEP];
    int n = 0;
    for (int h = threadIdx.x; h < H4; h += blockDim.x, ++n) {
        float4 s = extra ? extra[(size_t)t * H4 + h] : make_float4(0.f, 0.f, 0.f, 0.f);
        // every route's load issued first, then the sum in route order (a dropped route, id -1
        // under a load threshold, is skipped)
        float4 v[MOE_MAX_K];
        bool use[MOE_MAX_K];
#pragma unroll
        for (int j = 0; j < MOE_MAX_K; ++j) {
            use[j] = j < k && !(ids && ids[(size_t)t * k + j] < 0);
            if (use[j]) v[j] = partial[((size_t)t * k + j) * H4 + h];
        }
#pragma unroll
        for (int j = 0; j < MOE_MAX_K; ++j)
            if (use[j]) {
                s.x += v[j].x; s.y += v[j].y; s.z += v[j].z; s.w += v[j].w;
            }
        if (y) y[(size_t)t * H4 + h] = s;
        ss += s.x * s.x + s.y * s.y + s.z * s.z + s.w * s.w;
#pragma unroll
        for (int i = 0; i < KEEP; ++i)
            if (i == n) keep[i] = s;
        if (xn && n >= KEEP) xn[(size_t)t * H4 + h] = s;  // scaled below
    }
    if (!xn) return;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
    const float inv = 1.0f / sqrtf(tot / (float)(4 * H4) + eps);
    n = 0;
    for (int h = threadIdx.x; h < H4; h += blockDim.x, ++n) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (n < KEEP) {
#pragma unroll
            for (int i = 0; i < KEEP; ++i)
                if (i == n) v = keep[i];
        } else {
            v = xn[(size_t)t * H4 + h];
        }
        v.x *= inv; v.y *= inv; v.z *= inv; v.w *= inv;
        xn[(size_t)t * H4 + h] = v;
    }
}

// Resident CTAs of a ring kernel on the whole device at a dynamic shared-memory size,
// cached per (device, kernel, size).  The kernel's shared-memory limit is only ever raised,
// so every cached size stays launchable.
struct OccEntry {
    int dev;
    const void *fn;
    size_t smem;
    int ctas;
};

int ring_grid_capacity(const void *fn, size_t smem, int *ctas) {
    static std::mutex mu;
    static OccEntry tab[64];
    static int n_tab = 0;
    static struct { int dev; const void *fn; size_t max; } lim[32];
    static int n_lim = 0;
    int dev = 0;
    MOE_TRY_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < n_tab; ++i)
        if (tab[i].dev == dev && tab[i].fn == fn && tab[i].smem == smem) {
            *ctas = tab[i].ctas;
            return MOE_OK;
        }
    int li = -1;
    for (int i = 0; i < n_lim; ++i)
        if (lim[i].dev == dev && lim[i].fn == fn) li = i;
    if (li < 0 || lim[li].max < smem) {
        MOE_TRY_CUDA(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        if (li < 0 && n_lim < 32) li = n_lim++;
        if (li >= 0) lim[li] = {dev, fn, smem};
    }
    int occ = 0, sms = 0;
    MOE_TRY_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, GV_THREADS, smem));
    MOE_TRY_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    if (occ < 1 || sms < 1) return MOE_ERR_UNSUPPORTED;
    *ctas = std::min(occ * sms, GV_MAX_GRID);
    if (n_tab < 64) tab[n_tab++] = {dev, fn, smem, *ctas};
    return MOE_OK;
}

template <int QT, int XT, bool DOWN, int NTL>
const void *warp_fn() {
    return (const void *)ffn_warp_kernel<QT, XT, DOWN, NTL>;
}

// The GEMV kernel of a launch: G1 takes x as fp32 or bf16 and two tiles per unit; G2 takes
// fp32 activations and one or two tiles per unit.
const void *gemv_kernel_for(int qtype, int xtype, bool down, int ntl) {
    if (qtype == MOE_Q8_0) {
        if (down) return ntl == 2 ? warp_fn<MOE_Q8_0, MOE_F32, true, 2>() : warp_fn<MOE_Q8_0, MOE_F32, true, 1>();
        return xtype == MOE_F32 ? warp_fn<MOE_Q8_0, MOE_F32, false, 2>() : warp_fn<MOE_Q8_0, MOE_BF16, false, 2>();
    }
    if (down) return ntl == 2 ? warp_fn<MOE_Q4_SM, MOE_F32, true, 2>() : warp_fn<MOE_Q4_SM, MOE_F32, true, 1>();
    return xtype == MOE_F32 ? warp_fn<MOE_Q4_SM, MOE_F32, false, 2>() : warp_fn<MOE_Q4_SM, MOE_BF16, false, 2>();
}

template <int QT, int XT, int NTL2>
const void *fused_fn() {
    return (const void *)ffn_fused_kernel<QT, XT, NTL2>;
}

const void *fused_kernel_for(int qtype, int xtype, int ntl2) {
    if (qtype == MOE_Q8_0) {
        if (xtype == MOE_F32) return ntl2 == 2 ? fused_fn<MOE_Q8_0, MOE_F32, 2>() : fused_fn<MOE_Q8_0, MOE_F32, 1>();
        return ntl2 == 2 ? fused_fn<MOE_Q8_0, MOE_BF16, 2>() : fused_fn<MOE_Q8_0, MOE_BF16, 1>();
    }
    if (xtype == MOE_F32) return ntl2 == 2 ? fused_fn<MOE_Q4_SM, MOE_F32, 2>() : fused_fn<MOE_Q4_SM, MOE_F32, 1>();
    return ntl2 == 2 ? fused_fn<MOE_Q4_SM, MOE_BF16, 2>() : fused_fn<MOE_Q4_SM, MOE_BF16, 1>();
}

// Process-wide choice between the fused GEMV launch and the separate kernels.
std::atomic<int> g_fused{0};
// Whether a cooperative launch also takes the programmatic-dependency attribute (learnt at the
// first fused launch: 1 yes, 0 no, -1 not tried).
std::atomic<int> g_coop_pdl{-1};

}  // namespace

// A launch whose CTAs wait on one another: cooperative (the driver refuses a grid that cannot
// be resident at once), with the programmatic dependency on the previous kernel when the
// driver takes both attributes together.
static int launch_cooperative(const void *fn, dim3 grid, size_t smem, cudaStream_t s, void **args, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    moe_pdl_config(&cfg, attr, grid, dim3(GV_THREADS), smem, s);
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    const int mode = pdl ? g_coop_pdl.load() : 0;
    if (mode != 0) {
        cfg.numAttrs = 2;
        const cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
        if (e == cudaSuccess) {
            g_coop_pdl.store(1);
            return MOE_OK;
        }
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (mode == 1 || cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
            moe_note_cuda_error(e);
            return MOE_ERR_CUDA;
        }
        (void)cudaGetLastError();  // the combination was refused: launch cooperative alone
        g_coop_pdl.store(0);
    }
    cfg.attrs = attr + 1;
    cfg.numAttrs = 1;
    MOE_TRY_CUDA(cudaLaunchKernelExC(&cfg, fn, args));
    return MOE_OK;
}

extern "C" int moe_set_decode_fused(int on) {
    g_fused.store(on ? 1 : 0);
    return MOE_OK;
}

extern "C" int moe_get_decode_fused(void) { return g_fused.load(); }

int moe_decode_ffn_launches(int T, int H, int F, int qtype, int E, int k) {
    GvPlan pl;
    if (T <= 0 || !gv_plan(T, H, F, qtype, gv_n_act_max(T, E, k), &pl)) return 0;
    if (g_fused.load()) return 2;  // permute, fused gate/up + down
    return pl.KS > 1 ? 4 : 3;       // permute, gate/up, (K-split reduce,) down
}

size_t moe_decode_workspace_bytes(int T, int H, int F, int qtype, int E, int k) {
    // larger calls run in blocks of MOE_DECODE_MAX_T tokens that reuse one workspace
    return ws_layout(std::min(T, MOE_DECODE_MAX_T), H, F, qtype, E, k).total;
}

size_t moe_ffn_workspace_bytes(int T, int H, int F, int qtype, int xtype, int E, int k) {
    if (moe_prefill_eligible(T, H, F, qtype, xtype)) return moe_prefill_workspace_bytes(T, H, F, E, k);
    return moe_decode_workspace_bytes(T, H, F, qtype, E, k);
}

int moe_expert_ffn_impl(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k,
                        const int32_t *ids, const float *weights, const int32_t *d_slot_table,
                        int n_slots, const void *pool, size_t slot_bytes,
                        const int32_t *expert_subset, int n_subset, float *partial,
                        void *workspace, size_t ws_bytes, cudaStream_t s,
                        const moe_ffn_timing *timing) {
    return moe_expert_ffn_core(x, xtype, T, H, F, qtype, E, k, ids, weights, d_slot_table, n_slots, pool,
                               slot_bytes, expert_subset, n_subset, nullptr, partial, workspace, ws_bytes, s,
                               timing);
}

int moe_expert_ffn_core(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k,
                        const int32_t *ids, const float *weights, const int32_t *d_slot_table,
                        int n_slots, const void *pool, size_t slot_bytes,
                        const int32_t *expert_subset, int n_subset, const uint64_t *d_fill_src,
                        float *partial, void *workspace, size_t ws_bytes, cudaStream_t s,
                        const moe_ffn_timing *timing) {
    return moe_expert_ffn_stages(x, xtype, T, H, F, qtype, E, k, ids, weights, d_slot_table, n_slots, pool,
                                 slot_bytes, expert_subset, n_subset, d_fill_src, partial, workspace, ws_bytes, s,
                                 timing, MOE_FFN_ALL);
}

int moe_expert_ffn_stages(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k,
                          const int32_t *ids, const float *weights, const int32_t *d_slot_table,
                          int n_slots, const void *pool, size_t slot_bytes,
                          const int32_t *expert_subset, int n_subset, const uint64_t *d_fill_src,
                          float *partial, void *workspace, size_t ws_bytes, cudaStream_t s,
                          const moe_ffn_timing *timing, int stages) {
    MOE_CHECK(T >= 0);
    MOE_CHECK(qtype == MOE_Q8_0 || qtype == MOE_Q4_SM);
    MOE_CHECK(xtype == MOE_F32 || xtype == MOE_BF16);
    MOE_CHECK(H > 0 && F > 0 && H % 32 == 0 && F % 32 == 0);
    MOE_CHECK(E >= 1 && E <= MOE_MAX_E && k >= 1 && k <= MOE_MAX_K && k <= E);
    MOE_CHECK(n_subset >= 0 && n_subset <= E);
    if (T == 0 || (expert_subset && n_subset == 0)) return MOE_OK;
    MOE_CHECK(x && ids && weights && pool && partial && workspace);
    MOE_CHECK(n_slots >= 1);
    MOE_CHECK(((uintptr_t)pool & 15) == 0 && (slot_bytes & 15) == 0);
    MOE_CHECK(slot_bytes >= moe_expert_image_bytes(qtype, H, F));
    MOE_CHECK(((uintptr_t)workspace & 255) == 0);
    if (moe_prefill_eligible(T, H, F, qtype, xtype)) {
        if (d_fill_src || stages != MOE_FFN_ALL) return MOE_ERR_UNSUPPORTED;  // decode-path features
        MOE_CHECK(ws_bytes >= moe_prefill_workspace_bytes(T, H, F, E, k));
        return moe_prefill_ffn(x, xtype, T, H, F, qtype, E, k, ids, weights, d_slot_table, n_slots, pool,
                               slot_bytes, expert_subset, n_subset, partial, workspace, ws_bytes, s, timing);
    }
    if ((size_t)T * k > (1u << 20)) return MOE_ERR_UNSUPPORTED;
    if (T > MOE_DECODE_MAX_T) {  // token blocks of the decode size, one after another
        if (stages != MOE_FFN_ALL) return MOE_ERR_UNSUPPORTED;
        const size_t xb = xtype == MOE_F32 ? 4 : 2;
        for (int t0 = 0; t0 < T; t0 += MOE_DECODE_MAX_T) {
            const int Tb = std::min(MOE_DECODE_MAX_T, T - t0);
            const int rc = moe_expert_ffn_core((const char *)x + (size_t)t0 * H * xb, xtype, Tb, H, F, qtype, E, k,
                                               ids + (size_t)t0 * k, weights + (size_t)t0 * k, d_slot_table,
                                               n_slots, pool, slot_bytes, expert_subset, n_subset, d_fill_src,
                                               partial + (size_t)t0 * k * H, workspace, ws_bytes, s,
                                               t0 == 0 ? timing : nullptr);
            if (rc != MOE_OK) return rc;
        }
        return MOE_OK;
    }
    if (T * k > GV_PERMUTE_MAX_R) return MOE_ERR_UNSUPPORTED;
    const WsLayout W = ws_layout(T, H, F, qtype, E, k);
    MOE_CHECK(ws_bytes >= W.total);
    GvPlan pl;  // planned for every expert routable (the workspace does not depend on a subset)
    if (!gv_plan(T, H, F, qtype, gv_n_act_max(T, E, k), &pl)) return MOE_ERR_UNSUPPORTED;
    const int RTF = F / 32, RTH = H / 32;
    const size_t smem1 = gv_smem_bytes(pl.g1), smem2 = gv_smem_bytes(pl.g2);
    const void *k1 = gemv_kernel_for(qtype, xtype, false, 2), *k2 = gemv_kernel_for(qtype, xtype, true, pl.TPU);
    int cap1 = 0, cap2 = 0, rc;
    if ((rc = ring_grid_capacity(k1, smem1, &cap1)) != MOE_OK) return rc;
    if ((rc = ring_grid_capacity(k2, smem2, &cap2)) != MOE_OK) return rc;
    const int n_act_max = expert_subset ? n_subset : gv_n_act_max(T, E, k);
    const long n_virt_max = n_act_max + (long)T * k / GV_TOK + 1;
    const int per_v1 = pl.KS * RTF, per_v2 = RTH / pl.TPU;
    // One grid for both GEMVs, so that the permute kernel's unit ranges serve the fused launch
    // and the separate kernels alike.
    const void *kf = fused_kernel_for(qtype, xtype, pl.TPU);
    const size_t smemf = std::max(smem1, smem2);
    int capf = 0;
    if ((rc = ring_grid_capacity(kf, smemf, &capf)) != MOE_OK) return rc;
    const int cap = std::min(std::min(cap1, cap2), capf);
    // the gate/up launch gives each of its KS K ranges the same number of CTAs
    const int G0 = (int)std::max(1L, std::min((long)cap, n_virt_max * std::max(per_v1, per_v2)));
    const int G1 = std::max(pl.KS, G0 / pl.KS * pl.KS);
    const int G2 = G1;
    if (G1 > cap) return MOE_ERR_UNSUPPORTED;

    FfnParams p;
    p.x = x;
    p.T = T; p.H = H; p.F = F; p.k = k; p.E = E;
    p.KS = pl.KS;
    p.TPU = pl.TPU;
    p.RT = T * k;
    p.weights = weights;
    p.ws_ints = (const int32_t *)((char *)workspace + W.ints_off);
    p.info = (const ActInfo *)((char *)workspace + W.info_off);
    p.gu = (float *)((char *)workspace + W.gu_off);
    p.h = (float *)((char *)workspace + W.h_off);
    p.partial = partial;
    p.status = moe_status_word_device_ptr();
    p.x_vec = ((uintptr_t)x & 15) == 0;
    p.sync_extra = 0;
    p.sync_wait_ns = GV_GRID_WAIT_NS;

    if (stages & MOE_FFN_PERMUTE) {
    if (timing && timing->permute0) MOE_TRY_CUDA(cudaEventRecord(timing->permute0, s));
    {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        moe_pdl_config(&cfg, attr, dim3(1), dim3(256), 0, s);
        MOE_TRY_CUDA(cudaLaunchKernelEx(&cfg, permute_kernel, ids, T * k, E, expert_subset, n_subset,
                                        (int32_t *)((char *)workspace + W.ints_off),
                                        (ActInfo *)((char *)workspace + W.info_off), d_slot_table, n_slots,
                                        (const uint8_t *)pool, slot_bytes,
                                        (const unsigned long long *)d_fill_src, G1, per_v1, pl.KS, G2, per_v2,
                                        (unsigned long long *)((char *)workspace + W.first_off), p.status));
    }
    if (timing && timing->permute1) MOE_TRY_CUDA(cudaEventRecord(timing->permute1, s));
    }
    void *args[] = {&p};
    // The gate/up kernel reads x before its dependency wait.  Launched right behind this call's
    // permute kernel (which lets the next grid start only after its own wait, so everything
    // before it has completed) it may start early; otherwise only if the caller says x was
    // complete already, else behind a fully completed predecessor.
    const bool early_x = (stages & (MOE_FFN_PERMUTE | MOE_FFN_X_READY)) != 0;
    constexpr int kGemvStages = MOE_FFN_GATEUP | MOE_FFN_REDUCE | MOE_FFN_DOWN;
    if (g_fused.load() && (stages & kGemvStages) == kGemvStages) {
        if (timing && timing->gateup0) MOE_TRY_CUDA(cudaEventRecord(timing->gateup0, s));
        FfnParams p1 = p, p2 = p;
        if (moe_fault_take_grid_barrier()) {  // test fault injection: a barrier that times out
            p1.sync_extra = 1;
            p1.sync_wait_ns = GV_GRID_WAIT_TEST_NS;
        }
        p1.geo = pl.g1;
        p1.ranges = p.ws_ints + ws_ranges_off(E, T * k, 0);
        p1.first = (const unsigned long long *)((char *)workspace + W.first_off);
        p2.geo = pl.g2;
        p2.ranges = p.ws_ints + ws_ranges_off(E, T * k, 1);
        p2.first = p1.first + (size_t)GV_MAX_GRID * GV_WARPS;
        int *sync = (int *)((char *)workspace + W.ints_off) + GV_SYNC_OFF;
        void *fargs[] = {&p1, &p2, &sync};
        if ((rc = launch_cooperative(kf, dim3(G1), smemf, s, fargs, early_x)) != MOE_OK) return rc;
        if (timing && timing->gateup1) MOE_TRY_CUDA(cudaEventRecord(timing->gateup1, s));
        if (timing && timing->down0) MOE_TRY_CUDA(cudaEventRecord(timing->down0, s));
        if (timing && timing->down1) MOE_TRY_CUDA(cudaEventRecord(timing->down1, s));
        return MOE_OK;
    }
    if (stages & MOE_FFN_GATEUP) {
        if (timing && timing->gateup0) MOE_TRY_CUDA(cudaEventRecord(timing->gateup0, s));
        p.geo = pl.g1;
        p.ranges = p.ws_ints + ws_ranges_off(E, T * k, 0);
        p.first = (const unsigned long long *)((char *)workspace + W.first_off);
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        moe_pdl_config(&cfg, attr, dim3(G1), dim3(GV_THREADS), smem1, s);
        if (!early_x) cfg.numAttrs = 0;  // start only behind a completed predecessor
        MOE_TRY_CUDA(cudaLaunchKernelExC(&cfg, k1, args));
        if (timing && timing->gateup1 && !(stages & MOE_FFN_REDUCE)) MOE_TRY_CUDA(cudaEventRecord(timing->gateup1, s));
    }
    if ((stages & MOE_FFN_REDUCE) && pl.KS > 1) {  // h from the K-split partial sums
        const size_t n = (size_t)T * k * F;
        const int grid = (int)std::min<size_t>((n + 255) / 256, 4096);
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        moe_pdl_config(&cfg, attr, dim3(grid), dim3(256), 0, s);
        const float *gu = p.gu;
        float *h = p.h;
        switch (pl.KS) {
            case 2: MOE_TRY_CUDA(cudaLaunchKernelEx(&cfg, ks_reduce_kernel<2>, gu, h, n)); break;
            case 4: MOE_TRY_CUDA(cudaLaunchKernelEx(&cfg, ks_reduce_kernel<4>, gu, h, n)); break;
            case 8: MOE_TRY_CUDA(cudaLaunchKernelEx(&cfg, ks_reduce_kernel<8>, gu, h, n)); break;
            default: MOE_TRY_CUDA(cudaLaunchKernelEx(&cfg, ks_reduce_kernel<16>, gu, h, n)); break;
        }
    }
    if (stages & MOE_FFN_GATEUP) {
        if (timing && timing->gateup1 && (stages & MOE_FFN_REDUCE)) MOE_TRY_CUDA(cudaEventRecord(timing->gateup1, s));
    }
    if (stages & MOE_FFN_DOWN) {
        if (timing && timing->down0) MOE_TRY_CUDA(cudaEventRecord(timing->down0, s));
        p.geo = pl.g2;
        p.ranges = p.ws_ints + ws_ranges_off(E, T * k, 1);
        p.first = (const unsigned long long *)((char *)workspace + W.first_off) + (size_t)GV_MAX_GRID * GV_WARPS;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        moe_pdl_config(&cfg, attr, dim3(G2), dim3(GV_THREADS), smem2, s);
        MOE_TRY_CUDA(cudaLaunchKernelExC(&cfg, k2, args));
        if (timing && timing->down1) MOE_TRY_CUDA(cudaEventRecord(timing->down1, s));
    }
    return MOE_OK;
}

extern "C" int moe_expert_ffn(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k,
                              const int32_t *ids, const float *weights, const int32_t *d_slot_table,
                              int n_slots, const void *pool, size_t slot_bytes,
                              const int32_t *expert_subset, int n_subset, float *partial,
                              void *workspace, size_t ws_bytes, moe_stream_t s) {
    return moe_expert_ffn_impl(x, xtype, T, H, F, qtype, E, k, ids, weights, d_slot_table, n_slots,
                               pool, slot_bytes, expert_subset, n_subset, partial, workspace,
                               ws_bytes, moe_cuda_stream(s), nullptr);
}

extern "C" int moe_expert_ffn_fill(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k,
                                   const int32_t *ids, const float *weights, const int32_t *d_slot_table,
                                   int n_slots, void *pool, size_t slot_bytes, const uint64_t *d_fill_src,
                                   float *partial, void *workspace, size_t ws_bytes, moe_stream_t s) {
    MOE_CHECK(d_slot_table && d_fill_src);
    return moe_expert_ffn_core(x, xtype, T, H, F, qtype, E, k, ids, weights, d_slot_table, n_slots, pool,
                               slot_bytes, nullptr, 0, d_fill_src, partial, workspace, ws_bytes,
                               moe_cuda_stream(s), nullptr);
}

extern "C" int moe_expert_ffn_workspace(int T, int H, int F, int qtype, int xtype, int E, int k,
                                        size_t *bytes) {
    MOE_CHECK(bytes);
    MOE_CHECK(T >= 0 && H > 0 && F > 0 && H % 32 == 0 && F % 32 == 0);
    MOE_CHECK(qtype == MOE_Q8_0 || qtype == MOE_Q4_SM);
    MOE_CHECK(xtype == MOE_F32 || xtype == MOE_BF16);
    MOE_CHECK(E >= 1 && E <= MOE_MAX_E && k >= 1 && k <= MOE_MAX_K);
    *bytes = moe_ffn_workspace_bytes(T, H, F, qtype, xtype, E, k);
    return MOE_OK;
}

extern "C" int moe_combine_rmsnorm(const float *partial, int T, int k, int H, const float *extra, float *y,
                                   float *xn, float eps, moe_stream_t s) {
    return moe_combine_rmsnorm_routes(partial, nullptr, T, k, H, extra, y, xn, eps, moe_cuda_stream(s));
}

// moe_combine_rmsnorm skipping the routes whose id is -1 (ids [T][k] device, or NULL).
int moe_combine_rmsnorm_routes(const float *partial, const int32_t *ids, int T, int k, int H, const float *extra,
                               float *y, float *xn, float eps, cudaStream_t s) {
    MOE_CHECK(T >= 0 && k >= 0 && k <= 64 && H > 0 && H % 4 == 0 && eps >= 0.f);
    if (T == 0) return MOE_OK;
    MOE_CHECK(k == 0 || partial);
    MOE_CHECK(y || xn);
    MOE_CHECK(((uintptr_t)partial & 15) == 0 && ((uintptr_t)y & 15) == 0 && ((uintptr_t)extra & 15) == 0 &&
              ((uintptr_t)xn & 15) == 0);
    MOE_CHECK(!(xn && (xn == extra || xn == y)));
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    moe_pdl_config(&cfg, attr, dim3(T), dim3(256), 0, s);
    MOE_TRY_CUDA(cudaLaunchKernelEx(&cfg, combine_norm_kernel, (const float4 *)partial, k, H / 4,
                                    (const float4 *)extra, (float4 *)y, (float4 *)xn, eps, ids));
    return MOE_OK;
}

extern "C" int moe_combine(const float *partial, int T, int k, int H, const float *extra, float *y,
                           moe_stream_t s) {
    MOE_CHECK(T >= 0 && k >= 1 && k <= 64 && H > 0 && H % 4 == 0);
    if (T == 0) return MOE_OK;
    MOE_CHECK(partial && y);
    MOE_CHECK(((uintptr_t)partial & 15) == 0 && ((uintptr_t)y & 15) == 0 &&
              ((uintptr_t)extra & 15) == 0);
    const int H4 = H / 4;
    const size_t n = (size_t)T * H4;
    int grid = (int)((n + 255) / 256);
    if (grid > 152 * 8) grid = 152 * 8;
    combine_kernel<<<grid, 256, 0, moe_cuda_stream(s)>>>((const float4 *)partial, T, k, H4,
                                                          (const float4 *)extra, (float4 *)y);
    MOE_TRY_CUDA(cudaGetLastError());
    return MOE_OK;
}
