// TMA tensor-map construction (host).  All maps are bf16, row-major, with the
// 128-byte swizzle the GEMM engine's shared-memory descriptors expect, and zero
// fill outside the tensor (used for ragged token tails and for ranks below 64).
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace moelora {

// 2D tensor [outer][inner]; box of box_inner x box_outer elements.  Returns 0 on success.
int tmap_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
            uint32_t box_outer);
// 2D bf16 tensor [outer][inner] for epilogue TMA stores: 32 x 32 boxes (64-byte
// rows) with the 64-byte swizzle of the staging tiles (16-byte chunk j of row i
// sits at chunk j ^ ((i >> 1) & 3)).
int tmap_2d_store32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer);
// 3D tensor [d2][d1][d0]; box of b0 x b1 x 1.
int tmap_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1);
// 3D byte tensor [d2][d1][d0] (MXFP4 packed codes or scales), no swizzle: a box lands
// in shared memory as b1 rows of b0 bytes.  d0 a multiple of 16, b0 of 16.
int tmap_3d_u8(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1);

// bf16 tensor [d2][rows][cols] (cols % 64 == 0) seen as 64-column chunks -- dims
// {64, rows, cols/64, d2}, strides {cols*2, 128, rows*cols*2} bytes -- with a box of
// {64, 64, 4, 1}: one copy lands four MN-major 64 x 64 tiles of columns c0 .. c0+255,
// 8 KB apart, exactly as four 2D boxes would (chunks past the last column read zeros).
int tmap_mn4(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t d2);
// bf16 tensor [d2][rows][cols] (cols % 64 == 0, rows % 8 == 0) seen as {64 columns,
// 8 rows, cols/64 chunks, rows/8 groups, d2}; a box of {64, 8, chunks, 8, 1} lands 64
// rows x 64 chunks columns MN-major as 8-row groups (2 KB for two chunks) of 1 KB
// chunk atoms.
int tmap_mn_k8(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t d2, uint32_t chunks);
// 2D byte tensor [outer][inner] (E4M3 codes) with the 128-byte swizzle: a box of
// 128 x box_outer lands as box_outer rows of 128 bytes.
int tmap_2d_b8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer);
// E2M1 codes packed two per byte (low nibble first), [d2][d1][d0 codes] (d2 = 1 for
// a 2D tensor), copied to shared memory one code per byte position as the
// 16U4_ALIGN16B type does (each 16 codes = 8 bytes, then 8 bytes of gap) with the
// 128-byte swizzle; box 128 codes x b1 rows.  d0 a multiple of 128, base 32-byte
// aligned.
int tmap_fp4_unpacked(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b1);

}  // namespace moelora
