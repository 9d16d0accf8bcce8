// Host-side conversion between canonical expert tensors and slot images.
//
// Canonical tensors are page 2's expert-major ffn_{gate,up,down}_exps layout: one
// row per output feature, each row a run of quantised blocks along the reduction
// dimension.  The slot image (layout in moe_common.cuh) holds the same blocks
// regrouped: codes in 32-row tiles so that a warp's 16-byte loads are contiguous, each
// 32-column block's scales right after its codes (any K range of a tile is one run of
// bytes), and 8-bit codes in offset binary (q + 128).  Page 5 (section 1.2) keeps
// quantised blocks as they are on the GPU; so does this image (no dequantisation).
#include <string.h>

#include "moe_common.cuh"

namespace {

void pack_matrix(int qtype, int R, int K, const uint8_t *aos, uint8_t *dst) {
    const int NB = K / 32, BB = moe_block_bytes(qtype), SE = moe_scale_entry_bytes(qtype);
    for (int r = 0; r < R; ++r) {
        const int g = r / MOE_TILE_ROWS, lane = r % MOE_TILE_ROWS;
        for (int b = 0; b < NB; ++b) {
            const uint8_t *blk = aos + ((size_t)r * NB + b) * BB;
            uint8_t *tb = dst + moe_tile_block_offset(qtype, K, g, b);
            memcpy(tb + moe_scale_in_block(qtype, lane), blk, SE);
            if (qtype == MOE_Q8_0) {
                for (int half = 0; half < 2; ++half) {
                    uint8_t *q = tb + moe_piece_in_block(half, lane);
                    for (int i = 0; i < 16; ++i) q[i] = (uint8_t)(blk[2 + 16 * half + i] ^ 0x80);  // q + 128
                }
            } else {
                memcpy(tb + moe_piece_in_block(0, lane), blk + 4, 16);
            }
        }
    }
}

void unpack_matrix(int qtype, int R, int K, const uint8_t *src, uint8_t *aos) {
    const int NB = K / 32, BB = moe_block_bytes(qtype), SE = moe_scale_entry_bytes(qtype);
    for (int r = 0; r < R; ++r) {
        const int g = r / MOE_TILE_ROWS, lane = r % MOE_TILE_ROWS;
        for (int b = 0; b < NB; ++b) {
            uint8_t *blk = aos + ((size_t)r * NB + b) * BB;
            const uint8_t *tb = src + moe_tile_block_offset(qtype, K, g, b);
            memcpy(blk, tb + moe_scale_in_block(qtype, lane), SE);
            if (qtype == MOE_Q8_0) {
                for (int half = 0; half < 2; ++half) {
                    const uint8_t *q = tb + moe_piece_in_block(half, lane);
                    for (int i = 0; i < 16; ++i) blk[2 + 16 * half + i] = (uint8_t)(q[i] ^ 0x80);
                }
            } else {
                memcpy(blk + 4, tb + moe_piece_in_block(0, lane), 16);
            }
        }
    }
}

bool shape_ok(int qtype, int H, int F) {
    return (qtype == MOE_Q8_0 || qtype == MOE_Q4_SM) && H > 0 && F > 0 && H % 32 == 0 &&
           F % 32 == 0;
}

}  // namespace

extern "C" int moe_slot_image_bytes(int qtype, int H, int F, size_t *bytes_out) {
    MOE_CHECK(bytes_out && shape_ok(qtype, H, F));
    *bytes_out = moe_expert_image_bytes(qtype, H, F);
    return MOE_OK;
}

extern "C" int moe_pack_expert(int qtype, int H, int F, const void *gate_aos, const void *up_aos,
                               const void *down_aos, void *slot_image_dst, size_t *slot_bytes_out) {
    MOE_CHECK(shape_ok(qtype, H, F));
    const size_t total = moe_expert_image_bytes(qtype, H, F);
    if (slot_bytes_out) *slot_bytes_out = total;
    if (!slot_image_dst) return MOE_OK;
    MOE_CHECK(gate_aos && up_aos && down_aos);
    MOE_CHECK(((uintptr_t)slot_image_dst & 15) == 0);
    uint8_t *dst = (uint8_t *)slot_image_dst;
    pack_matrix(qtype, F, H, (const uint8_t *)gate_aos, dst + moe_expert_matrix_offset(qtype, H, F, 0));
    pack_matrix(qtype, F, H, (const uint8_t *)up_aos, dst + moe_expert_matrix_offset(qtype, H, F, 1));
    pack_matrix(qtype, H, F, (const uint8_t *)down_aos, dst + moe_expert_matrix_offset(qtype, H, F, 2));
    return MOE_OK;
}

extern "C" int moe_unpack_expert(int qtype, int H, int F, const void *slot_image, void *gate_aos,
                                 void *up_aos, void *down_aos) {
    MOE_CHECK(shape_ok(qtype, H, F));
    MOE_CHECK(slot_image && gate_aos && up_aos && down_aos);
    const uint8_t *src = (const uint8_t *)slot_image;
    unpack_matrix(qtype, F, H, src + moe_expert_matrix_offset(qtype, H, F, 0), (uint8_t *)gate_aos);
    unpack_matrix(qtype, F, H, src + moe_expert_matrix_offset(qtype, H, F, 1), (uint8_t *)up_aos);
    unpack_matrix(qtype, H, F, src + moe_expert_matrix_offset(qtype, H, F, 2), (uint8_t *)down_aos);
    return MOE_OK;
}
