// Compiled variants of the GEMV with binary16 weights and an FP32 x (the
// hidden state kept in FP32, "llama.cpp GEMV CUDA", implementation note).
// The FP32 x takes FP32 arithmetic: weights converted, x used as is.
#include "gemv_kernels.cuh"

namespace mbg {

static const Variant kTableF16X32[] = {
    // row bands (x in registers) for rows they cover exactly, the FP16 row
    // bands' shapes: band_t<threads>_c<chunks per thread>_g<rows per tile>_w<tiles in flight>
    MBG_BAND(DT_F16X32, 896, 2, 2, 2, 1, "band_t896_c2_g2_w2"),
    MBG_BAND(DT_F16X32, 256, 2, 2, 4, 2, "band_t256_c2_g2_w4"),
    MBG_BAND(DT_F16X32, 512, 4, 2, 2, 1, "band_t512_c4_g2_w2"),
    MBG_BAND(DT_F16X32, 448, 4, 2, 2, 1, "band_t448_c4_g2_w2"),
    MBG_TILE(DT_F16X32, 1, 8, 256, XMODE_BULK, "tile_g1_c8_t256_bulk"),
    MBG_TILE(DT_F16X32, 2, 8, 256, XMODE_BULK, "tile_g2_c8_t256_bulk"),
    MBG_TILE(DT_F16X32, 4, 8, 256, XMODE_BULK, "tile_g4_c8_t256_bulk"),
    MBG_TILE(DT_F16X32, 8, 8, 256, XMODE_BULK, "tile_g8_c8_t256_bulk"),
    MBG_TILE(DT_F16X32, 16, 8, 256, XMODE_BULK, "tile_g16_c8_t256_bulk"),
    MBG_TILE(DT_F16X32, 32, 8, 256, XMODE_BULK, "tile_g32_c8_t256_bulk"),
    MBG_TILE(DT_F16X32, 64, 8, 256, XMODE_BULK, "tile_g64_c8_t256_bulk"),
    MBG_TILE(DT_F16X32, 128, 8, 256, XMODE_BULK, "tile_g128_c8_t256_bulk"),
    MBG_TILE(DT_F16X32, 256, 8, 256, XMODE_BULK, "tile_g256_c8_t256_bulk"),
    MBG_TILE(DT_F16X32, 512, 8, 512, XMODE_BULK, "tile_g512_c8_t512_bulk"),
    MBG_TILE(DT_F16X32, 128, 8, 256, XMODE_L1, "tile_g128_c8_t256_l1"),
    MBG_TILE(DT_F16X32, 256, 8, 256, XMODE_L1, "tile_g256_c8_t256_l1"),
    MBG_TILE(DT_F16X32, 512, 8, 512, XMODE_L1, "tile_g512_c8_t512_l1"),
    MBG_BULK(DT_F16X32, 256, 1, 3, "bulk_t256_r1_s3"),
    MBG_BULK(DT_F16X32, 256, 4, 4, "bulk_t256_r4_s4"),
    MBG_VEC(DT_F16X32, 32, 1, 8, 4, XMODE_BULK, "w32_r1_u8_w4_bulk"),
    MBG_VEC(DT_F16X32, 32, 1, 8, 8, XMODE_L1, "w32_r1_u8_w8_l1"),
    MBG_ELEM(DT_F16X32, 4, "elem_w4"),
};

const Variant *variants_f16x32(int *count)
{
    *count = static_cast<int>(sizeof(kTableF16X32) / sizeof(kTableF16X32[0]));
    return kTableF16X32;
}

}  // namespace mbg
