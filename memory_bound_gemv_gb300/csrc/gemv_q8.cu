// Compiled variants of the q8 GEMV kernels.
//   bulk_t<consumer threads>_r<rows per stage>_s<pipeline stages>
//   tile_g<threads per row>_c<chunks per thread>_t<block threads>_<x staging>
//   w<lanes per row>_r<rows per group>_u<loads in flight>_w<warps>_<x staging>
#include "gemv_kernels.cuh"

namespace mbg {

static const Variant kTableQ8[] = {
    // the automatic choice takes, in table order, the first row band or
    // fixed-count bulk pipeline that covers the row exactly (measured best first)
    // MMA row bands (products on the MMA unit), mma_w<warps>_s<steps per
    // warp>_t<tiles in flight>_m<min blocks per SM>: rows of exactly warps *
    // steps * 512 bytes (measured best of every design at 4096 and 14336 columns)
    MBG_MMA(DT_Q8, 8, 1, 4, 2, "mma_w8_s1_t4_m2"),
    MBG_MMA(DT_Q8, 28, 1, 2, 1, "mma_w28_s1_t2_m1"),
    MBG_BAND(DT_Q8, 256, 1, 2, 4, 2, "band_t256_c1_g2_w4"),
    // bulk-copy pipelines specialised for rows of exactly f * t chunks:
    // bulk_t<consumer threads>_r<rows per stage>_s<stages>_f<chunks per thread>
    MBG_BULK_F(DT_Q8, 128, 4, 3, 2, "bulk_t128_r4_s3_f2"),
    MBG_BULK_FX(DT_Q8, 224, 1, 3, 4, "bulk_t224_r1_s3_f4_xr"),
    MBG_BULK_F(DT_Q8, 224, 1, 3, 4, "bulk_t224_r1_s3_f4"),
    MBG_BULK_F(DT_Q8, 128, 4, 2, 2, "bulk_t128_r4_s2_f2"),
    // other row bands (x in registers), band_t<threads>_c<chunks per thread>_g<rows per tile>_w<tiles in flight>
    MBG_BAND(DT_Q8, 256, 1, 4, 4, 1, "band_t256_c1_g4_w4"),
    MBG_BAND(DT_Q8, 128, 2, 2, 4, 3, "band_t128_c2_g2_w4"),
    MBG_BAND(DT_Q8, 448, 2, 2, 2, 1, "band_t448_c2_g2_w2"),
    MBG_BAND(DT_Q8, 896, 1, 2, 2, 1, "band_t896_c1_g2_w2"),
    MBG_BAND(DT_Q8, 224, 4, 2, 2, 1, "band_t224_c4_g2_w2"),
    // staged row bands (tiles of A in shared memory by bulk copies):
    // sband_t<threads>_c<chunks per thread>_g<rows per tile>_w<tiles per window>_p<windows in flight>
    MBG_SBAND(DT_Q8, 256, 1, 2, 2, 1, 4, "sband_t256_c1_g2_w2_p1"),
    MBG_SBAND(DT_Q8, 256, 1, 2, 2, 2, 3, "sband_t256_c1_g2_w2_p2"),
    MBG_SBAND(DT_Q8, 128, 2, 2, 4, 2, 3, "sband_t128_c2_g2_w4_p2"),
    MBG_SBAND(DT_Q8, 448, 2, 2, 2, 1, 1, "sband_t448_c2_g2_w2_p1"),
    MBG_SBAND(DT_Q8, 448, 2, 1, 2, 2, 1, "sband_t448_c2_g1_w2_p2"),
    MBG_SBAND(DT_Q8, 896, 1, 1, 2, 2, 1, "sband_t896_c1_g1_w2_p2"),
    // other MMA row bands (explicit choice)
    MBG_MMA(DT_Q8, 8, 1, 2, 4, "mma_w8_s1_t2_m4"),
    MBG_MMA(DT_Q8, 4, 2, 2, 4, "mma_w4_s2_t2_m4"),
    MBG_MMA(DT_Q8, 14, 2, 2, 2, "mma_w14_s2_t2_m2"),
    // the same with row-contiguous loads
    MBG_MMA_L(DT_Q8, 8, 1, 4, 2, true, "mma_w8_s1_t4_m2_rc"),
    MBG_MMA_L(DT_Q8, 28, 1, 2, 1, true, "mma_w28_s1_t2_m1_rc"),
    // staged MMA row bands, smma_w<warps>_s<steps per warp>_r<row pairs per
    // tile>_t<tiles per window>_p<windows in flight>_m<min blocks per SM>:
    // rows of exactly warps * steps * 512 bytes (explicit choice)
    MBG_SMMA(DT_Q8, 8, 1, 2, 2, 2, 2, "smma_w8_s1_r2_t2_p2_m2"),
    MBG_SMMA(DT_Q8, 14, 2, 1, 2, 2, 1, "smma_w14_s2_r1_t2_p2_m1"),
    // general variants (explicit choice, and the fallbacks of the automatic one)
    // bulk-copy pipelines: bulk_t<consumer threads>_r<rows per stage>_s<stages>
    MBG_BULK(DT_Q8, 256, 1, 3, "bulk_t256_r1_s3"),
    MBG_BULK(DT_Q8, 256, 1, 4, "bulk_t256_r1_s4"),
    MBG_BULK(DT_Q8, 512, 1, 4, "bulk_t512_r1_s4"),
    MBG_BULK(DT_Q8, 256, 2, 4, "bulk_t256_r2_s4"),
    MBG_BULK(DT_Q8, 512, 2, 4, "bulk_t512_r2_s4"),
    MBG_BULK(DT_Q8, 256, 4, 4, "bulk_t256_r4_s4"),
    MBG_BULK(DT_Q8, 512, 4, 4, "bulk_t512_r4_s4"),
    MBG_BULK(DT_Q8, 256, 8, 3, "bulk_t256_r8_s3"),
    MBG_BULK(DT_Q8, 512, 8, 4, "bulk_t512_r8_s4"),
    MBG_BULK(DT_Q8, 128, 4, 2, "bulk_t128_r4_s2"),
    // row tiles (the automatic choice for rows up to 512 * 8 * 16 bytes)
    MBG_TILE(DT_Q8, 1, 8, 256, XMODE_BULK, "tile_g1_c8_t256_bulk"),
    MBG_TILE(DT_Q8, 2, 8, 256, XMODE_BULK, "tile_g2_c8_t256_bulk"),
    MBG_TILE(DT_Q8, 4, 8, 256, XMODE_BULK, "tile_g4_c8_t256_bulk"),
    MBG_TILE(DT_Q8, 8, 8, 256, XMODE_BULK, "tile_g8_c8_t256_bulk"),
    MBG_TILE(DT_Q8, 16, 8, 256, XMODE_BULK, "tile_g16_c8_t256_bulk"),
    MBG_TILE(DT_Q8, 32, 8, 256, XMODE_BULK, "tile_g32_c8_t256_bulk"),
    MBG_TILE(DT_Q8, 64, 8, 256, XMODE_BULK, "tile_g64_c8_t256_bulk"),
    MBG_TILE(DT_Q8, 128, 8, 256, XMODE_BULK, "tile_g128_c8_t256_bulk"),
    MBG_TILE(DT_Q8, 256, 8, 256, XMODE_BULK, "tile_g256_c8_t256_bulk"),
    MBG_TILE(DT_Q8, 512, 8, 512, XMODE_BULK, "tile_g512_c8_t512_bulk"),
    // row-tile alternatives (block size, x through L1)
    MBG_TILE(DT_Q8, 64, 8, 512, XMODE_BULK, "tile_g64_c8_t512_bulk"),
    MBG_TILE(DT_Q8, 128, 8, 512, XMODE_BULK, "tile_g128_c8_t512_bulk"),
    MBG_TILE(DT_Q8, 256, 8, 512, XMODE_BULK, "tile_g256_c8_t512_bulk"),
    MBG_TILE(DT_Q8, 512, 4, 512, XMODE_BULK, "tile_g512_c4_t512_bulk"),
    MBG_TILE(DT_Q8, 256, 4, 256, XMODE_BULK, "tile_g256_c4_t256_bulk"),
    MBG_TILE(DT_Q8, 64, 8, 256, XMODE_L1, "tile_g64_c8_t256_l1"),
    MBG_TILE(DT_Q8, 128, 8, 256, XMODE_L1, "tile_g128_c8_t256_l1"),
    MBG_TILE(DT_Q8, 256, 8, 256, XMODE_L1, "tile_g256_c8_t256_l1"),
    MBG_TILE(DT_Q8, 512, 8, 512, XMODE_L1, "tile_g512_c8_t512_l1"),
    // row tiles with operands converted to FP32 (for comparison)
    MBG_TILE_M(DT_Q8, 64, 8, 256, XMODE_BULK, MATH_F32, "tile_g64_c8_t256_bulk_f32math"),
    MBG_TILE_M(DT_Q8, 256, 8, 256, XMODE_BULK, MATH_F32, "tile_g256_c8_t256_bulk_f32math"),
    MBG_TILE_M(DT_Q8, 512, 4, 512, XMODE_BULK, MATH_F32, "tile_g512_c4_t512_bulk_f32math"),
    // rows of a warp (or of part of one) with a rolling buffer of loads
    MBG_VEC(DT_Q8, 32, 1, 8, 4, XMODE_BULK, "w32_r1_u8_w4_bulk"),
    MBG_VEC(DT_Q8, 32, 1, 4, 8, XMODE_BULK, "w32_r1_u4_w8_bulk"),
    MBG_VEC(DT_Q8, 32, 2, 4, 4, XMODE_BULK, "w32_r2_u4_w4_bulk"),
    MBG_VEC(DT_Q8, 32, 1, 8, 4, XMODE_VEC, "w32_r1_u8_w4_vec"),
    MBG_VEC(DT_Q8, 32, 1, 8, 8, XMODE_L1, "w32_r1_u8_w8_l1"),
    MBG_VEC(DT_Q8, 16, 1, 2, 4, XMODE_BULK, "w16_r1_u2_w4_bulk"),
    MBG_VEC(DT_Q8, 4, 1, 2, 4, XMODE_BULK, "w4_r1_u2_w4_bulk"),
    MBG_VEC(DT_Q8, 1, 1, 2, 4, XMODE_BULK, "w1_r1_u2_w4_bulk"),
    // any layout
    MBG_ELEM(DT_Q8, 4, "elem_w4"),
};

const Variant *variants_q8(int *count)
{
    *count = static_cast<int>(sizeof(kTableQ8) / sizeof(kTableQ8[0]));
    return kTableQ8;
}

}  // namespace mbg
