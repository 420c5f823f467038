// Compiled variants of the q4 GEMV kernels.
//   bulk_t<consumer threads>_r<rows per stage>_s<pipeline stages>
//   tile_g<threads per row>_c<chunks per thread>_t<block threads>_<x staging>
//   w<lanes per row>_r<rows per group>_u<loads in flight>_w<warps>_<x staging>
#include "gemv_kernels.cuh"

namespace mbg {

static const Variant kTableQ4[] = {
    // the automatic choice takes, in table order, the first row band, MMA row
    // band or fixed-count bulk pipeline that covers the row exactly (measured
    // best first)
    // MMA row band with row-contiguous loads, rows of 2048 bytes (4096 codes):
    // 8.1 us at 14336x4096 against 8.8 us for the bulk pipeline below
    MBG_MMA_L(DT_Q4, 4, 1, 4, 1, true, "mma_w4_s1_t4_m1_rc"),
    // bulk-copy pipelines specialised for rows of exactly f * t chunks:
    // bulk_t<consumer threads>_r<rows per stage>_s<stages>_f<chunks per thread>
    MBG_BULK_F(DT_Q4, 224, 2, 3, 2, "bulk_t224_r2_s3_f2"),
    MBG_BULK_F(DT_Q4, 128, 4, 3, 1, "bulk_t128_r4_s3_f1"),
    // other row bands (x in registers), band_t<threads>_c<chunks per thread>_g<rows per tile>_w<tiles in flight>
    MBG_BAND(DT_Q4, 128, 1, 4, 4, 3, "band_t128_c1_g4_w4"),
    MBG_BAND(DT_Q4, 128, 1, 2, 4, 4, "band_t128_c1_g2_w4"),
    MBG_BAND(DT_Q4, 64, 2, 4, 2, 5, "band_t64_c2_g4_w2"),
    MBG_BAND(DT_Q4, 448, 1, 2, 4, 1, "band_t448_c1_g2_w4"),
    MBG_BAND(DT_Q4, 448, 1, 4, 2, 1, "band_t448_c1_g4_w2"),
    MBG_BAND(DT_Q4, 224, 2, 2, 4, 1, "band_t224_c2_g2_w4"),
    MBG_BAND(DT_Q4, 128, 1, 2, 2, 6, "band_t128_c1_g2_w2"),
    MBG_BAND(DT_Q4, 128, 1, 4, 2, 5, "band_t128_c1_g4_w2"),
    MBG_BAND(DT_Q4, 448, 1, 2, 2, 2, "band_t448_c1_g2_w2"),
    // staged row bands (tiles of A in shared memory by bulk copies):
    // sband_t<threads>_c<chunks per thread>_g<rows per tile>_w<tiles per window>_p<windows in flight>
    MBG_SBAND(DT_Q4, 128, 1, 4, 2, 1, 6, "sband_t128_c1_g4_w2_p1"),
    MBG_SBAND(DT_Q4, 128, 1, 4, 2, 2, 4, "sband_t128_c1_g4_w2_p2"),
    MBG_SBAND(DT_Q4, 128, 1, 2, 4, 2, 4, "sband_t128_c1_g2_w4_p2"),
    MBG_SBAND(DT_Q4, 128, 1, 8, 2, 1, 3, "sband_t128_c1_g8_w2_p1"),
    MBG_SBAND(DT_Q4, 128, 1, 4, 2, 3, 3, "sband_t128_c1_g4_w2_p3"),
    MBG_SBAND(DT_Q4, 448, 1, 2, 2, 1, 2, "sband_t448_c1_g2_w2_p1"),
    MBG_SBAND(DT_Q4, 448, 1, 2, 2, 2, 1, "sband_t448_c1_g2_w2_p2"),
    MBG_SBAND(DT_Q4, 224, 2, 2, 2, 2, 3, "sband_t224_c2_g2_w2_p2"),
    MBG_SBAND(DT_Q4, 224, 2, 1, 4, 2, 3, "sband_t224_c2_g1_w4_p2"),
    // other MMA row bands (products on the MMA unit), mma_w<warps>_s<steps per
    // warp>_t<tiles in flight>_m<min blocks per SM>[_rc]: rows of exactly warps
    // * steps * 512 bytes (explicit choice: within noise of the bulk pipelines
    // at 14336 columns)
    MBG_MMA(DT_Q4, 14, 1, 4, 1, "mma_w14_s1_t4_m1"),
    MBG_MMA(DT_Q4, 4, 1, 4, 1, "mma_w4_s1_t4_m1"),
    MBG_MMA(DT_Q4, 4, 1, 4, 4, "mma_w4_s1_t4_m4"),
    MBG_MMA(DT_Q4, 14, 1, 2, 2, "mma_w14_s1_t2_m2"),
    // the same with row-contiguous loads
    MBG_MMA_L(DT_Q4, 14, 1, 4, 1, true, "mma_w14_s1_t4_m1_rc"),
    // staged MMA row bands, smma_w<warps>_s<steps per warp>_r<row pairs per
    // tile>_t<tiles per window>_p<windows in flight>_m<min blocks per SM>:
    // rows of exactly warps * steps * 512 bytes (explicit choice)
    MBG_SMMA(DT_Q4, 4, 1, 4, 2, 1, 3, "smma_w4_s1_r4_t2_p1_m3"),
    MBG_SMMA(DT_Q4, 14, 1, 2, 2, 1, 1, "smma_w14_s1_r2_t2_p1_m1"),
    MBG_SMMA(DT_Q4, 7, 2, 2, 2, 1, 2, "smma_w7_s2_r2_t2_p1_m2"),
    // general variants (explicit choice, and the fallbacks of the automatic one)
    MBG_BULK(DT_Q4, 256, 1, 4, "bulk_t256_r1_s4"),
    MBG_BULK(DT_Q4, 256, 1, 3, "bulk_t256_r1_s3"),
    MBG_BULK(DT_Q4, 512, 1, 4, "bulk_t512_r1_s4"),
    MBG_BULK(DT_Q4, 256, 2, 4, "bulk_t256_r2_s4"),
    MBG_BULK(DT_Q4, 512, 2, 4, "bulk_t512_r2_s4"),
    MBG_BULK(DT_Q4, 256, 4, 4, "bulk_t256_r4_s4"),
    MBG_BULK(DT_Q4, 512, 4, 4, "bulk_t512_r4_s4"),
    MBG_BULK(DT_Q4, 256, 8, 3, "bulk_t256_r8_s3"),
    MBG_BULK(DT_Q4, 512, 8, 4, "bulk_t512_r8_s4"),
    MBG_BULK(DT_Q4, 224, 2, 3, "bulk_t224_r2_s3"),
    // row tiles (the automatic choice for rows up to 512 * 8 * 16 bytes)
    MBG_TILE(DT_Q4, 1, 8, 256, XMODE_BULK, "tile_g1_c8_t256_bulk"),
    MBG_TILE(DT_Q4, 2, 8, 256, XMODE_BULK, "tile_g2_c8_t256_bulk"),
    MBG_TILE(DT_Q4, 4, 8, 256, XMODE_BULK, "tile_g4_c8_t256_bulk"),
    MBG_TILE(DT_Q4, 8, 8, 256, XMODE_BULK, "tile_g8_c8_t256_bulk"),
    MBG_TILE(DT_Q4, 16, 8, 256, XMODE_BULK, "tile_g16_c8_t256_bulk"),
    MBG_TILE(DT_Q4, 32, 8, 256, XMODE_BULK, "tile_g32_c8_t256_bulk"),
    MBG_TILE(DT_Q4, 64, 8, 256, XMODE_BULK, "tile_g64_c8_t256_bulk"),
    MBG_TILE(DT_Q4, 128, 8, 256, XMODE_BULK, "tile_g128_c8_t256_bulk"),
    MBG_TILE(DT_Q4, 256, 8, 256, XMODE_BULK, "tile_g256_c8_t256_bulk"),
    MBG_TILE(DT_Q4, 512, 8, 512, XMODE_BULK, "tile_g512_c8_t512_bulk"),
    // row-tile alternatives (block size, x through L1)
    MBG_TILE(DT_Q4, 64, 8, 512, XMODE_BULK, "tile_g64_c8_t512_bulk"),
    MBG_TILE(DT_Q4, 128, 8, 512, XMODE_BULK, "tile_g128_c8_t512_bulk"),
    MBG_TILE(DT_Q4, 256, 8, 512, XMODE_BULK, "tile_g256_c8_t512_bulk"),
    MBG_TILE(DT_Q4, 512, 4, 512, XMODE_BULK, "tile_g512_c4_t512_bulk"),
    MBG_TILE(DT_Q4, 256, 4, 256, XMODE_BULK, "tile_g256_c4_t256_bulk"),
    MBG_TILE(DT_Q4, 32, 4, 128, XMODE_BULK, "tile_g32_c4_t128_bulk"),
    MBG_TILE(DT_Q4, 64, 8, 256, XMODE_L1, "tile_g64_c8_t256_l1"),
    MBG_TILE(DT_Q4, 128, 8, 256, XMODE_L1, "tile_g128_c8_t256_l1"),
    MBG_TILE(DT_Q4, 256, 8, 256, XMODE_L1, "tile_g256_c8_t256_l1"),
    MBG_TILE(DT_Q4, 512, 8, 512, XMODE_L1, "tile_g512_c8_t512_l1"),
    // row tiles with operands converted to FP32 (for comparison)
    MBG_TILE_M(DT_Q4, 64, 8, 256, XMODE_BULK, MATH_F32, "tile_g64_c8_t256_bulk_f32math"),
    MBG_TILE_M(DT_Q4, 256, 8, 256, XMODE_BULK, MATH_F32, "tile_g256_c8_t256_bulk_f32math"),
    MBG_TILE_M(DT_Q4, 512, 4, 512, XMODE_BULK, MATH_F32, "tile_g512_c4_t512_bulk_f32math"),
    // rows of a warp (or of part of one) with a rolling buffer of loads
    MBG_VEC(DT_Q4, 32, 1, 8, 4, XMODE_BULK, "w32_r1_u8_w4_bulk"),
    MBG_VEC(DT_Q4, 32, 1, 4, 8, XMODE_BULK, "w32_r1_u4_w8_bulk"),
    MBG_VEC(DT_Q4, 32, 2, 4, 4, XMODE_BULK, "w32_r2_u4_w4_bulk"),
    MBG_VEC(DT_Q4, 32, 1, 8, 4, XMODE_VEC, "w32_r1_u8_w4_vec"),
    MBG_VEC(DT_Q4, 32, 1, 8, 8, XMODE_L1, "w32_r1_u8_w8_l1"),
    MBG_VEC(DT_Q4, 16, 1, 2, 4, XMODE_BULK, "w16_r1_u2_w4_bulk"),
    MBG_VEC(DT_Q4, 4, 1, 2, 4, XMODE_BULK, "w4_r1_u2_w4_bulk"),
    MBG_VEC(DT_Q4, 1, 1, 2, 4, XMODE_BULK, "w1_r1_u2_w4_bulk"),
    // any layout
    MBG_ELEM(DT_Q4, 4, "elem_w4"),
};

const Variant *variants_q4(int *count)
{
    *count = static_cast<int>(sizeof(kTableQ4) / sizeof(kTableQ4[0]));
    return kTableQ4;
}

}  // namespace mbg
