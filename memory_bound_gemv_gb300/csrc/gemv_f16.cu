// Compiled variants of the f16 GEMV kernels.
//   bulk_t<consumer threads>_r<rows per stage>_s<pipeline stages>
//   tile_g<threads per row>_c<chunks per thread>_t<block threads>_<x staging>
//   w<lanes per row>_r<rows per group>_u<loads in flight>_w<warps>_<x staging>
#include "gemv_kernels.cuh"

namespace mbg {

static const Variant kTableF16[] = {
    // row bands, x in registers: band_t<threads>_c<chunks per thread>_g<rows per
    // tile>_w<tiles in flight> (rows of exactly threads * chunks 16-byte chunks); for a given row
    // length the first that fits is the automatic choice (measured best first)
    MBG_BAND_CAP(DT_F16, 128, 2, 2, 4, 4, 2, "band_t128_c2_g2_w4_b2"),
    MBG_BAND(DT_F16, 256, 1, 2, 4, 2, "band_t256_c1_g2_w4"),
    MBG_BAND(DT_F16, 128, 2, 2, 4, 4, "band_t128_c2_g2_w4"),
    MBG_BAND(DT_F16, 256, 2, 2, 4, 2, "band_t256_c2_g2_w4"),
    MBG_BAND(DT_F16, 128, 4, 2, 2, 4, "band_t128_c4_g2_w2"),
    MBG_BAND(DT_F16, 256, 4, 2, 2, 2, "band_t256_c4_g2_w2"),
    MBG_BAND(DT_F16, 512, 2, 2, 2, 1, "band_t512_c2_g2_w2"),
    MBG_BAND(DT_F16, 896, 2, 2, 2, 1, "band_t896_c2_g2_w2"),
    MBG_BAND(DT_F16, 448, 4, 2, 2, 1, "band_t448_c4_g2_w2"),
    MBG_BAND(DT_F16, 512, 4, 2, 2, 1, "band_t512_c4_g2_w2"),
    // band_..._b<n>: at most n blocks per SM, so that the next launch's blocks fit beside them
    // (small matrices only)
    MBG_BAND_CAP(DT_F16, 256, 1, 2, 4, 2, 1, "band_t256_c1_g2_w4_b1"),
    MBG_BAND_CAP(DT_F16, 128, 2, 2, 2, 4, 2, "band_t128_c2_g2_w2_b2"),
    MBG_BAND_CAP(DT_F16, 256, 2, 2, 4, 2, 1, "band_t256_c2_g2_w4_b1"),
    // staged row bands (tiles of A in shared memory by bulk copies):
    // sband_t<threads>_c<chunks per thread>_g<rows per tile>_w<tiles per window>_p<windows in flight>
    MBG_SBAND(DT_F16, 256, 2, 2, 2, 1, 3, "sband_t256_c2_g2_w2_p1"),
    MBG_SBAND(DT_F16, 448, 4, 1, 2, 1, 1, "sband_t448_c4_g1_w2_p1"),
    // bulk-copy pipelines: bulk_t<consumer threads>_r<rows per stage>_s<stages>
    MBG_BULK(DT_F16, 256, 1, 4, "bulk_t256_r1_s4"),
    MBG_BULK(DT_F16, 256, 1, 3, "bulk_t256_r1_s3"),
    MBG_BULK(DT_F16, 512, 1, 4, "bulk_t512_r1_s4"),
    MBG_BULK(DT_F16, 256, 2, 4, "bulk_t256_r2_s4"),
    MBG_BULK(DT_F16, 512, 2, 4, "bulk_t512_r2_s4"),
    MBG_BULK(DT_F16, 256, 4, 4, "bulk_t256_r4_s4"),
    MBG_BULK(DT_F16, 512, 4, 4, "bulk_t512_r4_s4"),
    MBG_BULK(DT_F16, 256, 8, 3, "bulk_t256_r8_s3"),
    MBG_BULK(DT_F16, 512, 8, 4, "bulk_t512_r8_s4"),
    // row tiles (the automatic choice for rows up to 512 * 8 * 16 bytes)
    MBG_TILE(DT_F16, 1, 8, 256, XMODE_BULK, "tile_g1_c8_t256_bulk"),
    MBG_TILE(DT_F16, 2, 8, 256, XMODE_BULK, "tile_g2_c8_t256_bulk"),
    MBG_TILE(DT_F16, 4, 8, 256, XMODE_BULK, "tile_g4_c8_t256_bulk"),
    MBG_TILE(DT_F16, 8, 8, 256, XMODE_BULK, "tile_g8_c8_t256_bulk"),
    MBG_TILE(DT_F16, 16, 8, 256, XMODE_BULK, "tile_g16_c8_t256_bulk"),
    MBG_TILE(DT_F16, 32, 8, 256, XMODE_BULK, "tile_g32_c8_t256_bulk"),
    MBG_TILE(DT_F16, 64, 8, 256, XMODE_BULK, "tile_g64_c8_t256_bulk"),
    MBG_TILE(DT_F16, 128, 8, 256, XMODE_BULK, "tile_g128_c8_t256_bulk"),
    MBG_TILE(DT_F16, 256, 8, 256, XMODE_BULK, "tile_g256_c8_t256_bulk"),
    MBG_TILE(DT_F16, 512, 8, 512, XMODE_BULK, "tile_g512_c8_t512_bulk"),
    // row-tile alternatives (block size, x through L1)
    MBG_TILE(DT_F16, 64, 8, 512, XMODE_BULK, "tile_g64_c8_t512_bulk"),
    MBG_TILE(DT_F16, 128, 8, 512, XMODE_BULK, "tile_g128_c8_t512_bulk"),
    MBG_TILE(DT_F16, 256, 8, 512, XMODE_BULK, "tile_g256_c8_t512_bulk"),
    MBG_TILE(DT_F16, 512, 4, 512, XMODE_BULK, "tile_g512_c4_t512_bulk"),
    MBG_TILE(DT_F16, 256, 4, 256, XMODE_BULK, "tile_g256_c4_t256_bulk"),
    MBG_TILE(DT_F16, 64, 8, 256, XMODE_L1, "tile_g64_c8_t256_l1"),
    MBG_TILE(DT_F16, 128, 8, 256, XMODE_L1, "tile_g128_c8_t256_l1"),
    MBG_TILE(DT_F16, 256, 8, 256, XMODE_L1, "tile_g256_c8_t256_l1"),
    MBG_TILE(DT_F16, 512, 8, 512, XMODE_L1, "tile_g512_c8_t512_l1"),
    // 128-thread blocks (finer tiles, more blocks per SM)
    MBG_TILE(DT_F16, 16, 8, 128, XMODE_BULK, "tile_g16_c8_t128_bulk"),
    MBG_TILE(DT_F16, 32, 8, 128, XMODE_BULK, "tile_g32_c8_t128_bulk"),
    MBG_TILE(DT_F16, 32, 8, 128, XMODE_L1, "tile_g32_c8_t128_l1"),
    MBG_TILE(DT_F16, 64, 8, 128, XMODE_L1, "tile_g64_c8_t128_l1"),
    MBG_TILE(DT_F16, 64, 8, 128, XMODE_BULK, "tile_g64_c8_t128_bulk"),
    MBG_TILE(DT_F16, 128, 8, 128, XMODE_L1, "tile_g128_c8_t128_l1"),
    MBG_TILE(DT_F16, 128, 4, 128, XMODE_L1, "tile_g128_c4_t128_l1"),
    // row tiles with operands converted to FP32 (for comparison)
    MBG_TILE_M(DT_F16, 64, 8, 256, XMODE_BULK, MATH_F32, "tile_g64_c8_t256_bulk_f32math"),
    MBG_TILE_M(DT_F16, 256, 8, 256, XMODE_BULK, MATH_F32, "tile_g256_c8_t256_bulk_f32math"),
    MBG_TILE_M(DT_F16, 512, 4, 512, XMODE_BULK, MATH_F32, "tile_g512_c4_t512_bulk_f32math"),
    // rows of a warp (or of part of one) with a rolling buffer of loads
    MBG_VEC(DT_F16, 32, 1, 8, 4, XMODE_BULK, "w32_r1_u8_w4_bulk"),
    MBG_VEC(DT_F16, 32, 1, 4, 8, XMODE_BULK, "w32_r1_u4_w8_bulk"),
    MBG_VEC(DT_F16, 32, 2, 4, 4, XMODE_BULK, "w32_r2_u4_w4_bulk"),
    MBG_VEC(DT_F16, 32, 1, 8, 4, XMODE_VEC, "w32_r1_u8_w4_vec"),
    MBG_VEC(DT_F16, 32, 1, 8, 8, XMODE_L1, "w32_r1_u8_w8_l1"),
    MBG_VEC(DT_F16, 16, 1, 2, 4, XMODE_BULK, "w16_r1_u2_w4_bulk"),
    MBG_VEC(DT_F16, 4, 1, 2, 4, XMODE_BULK, "w4_r1_u2_w4_bulk"),
    MBG_VEC(DT_F16, 1, 1, 2, 4, XMODE_BULK, "w1_r1_u2_w4_bulk"),
    // any layout
    MBG_ELEM(DT_F16, 4, "elem_w4"),
};

const Variant *variants_f16(int *count)
{
    *count = static_cast<int>(sizeof(kTableF16) / sizeof(kTableF16[0]));
    return kTableF16;
}

}  // namespace mbg
