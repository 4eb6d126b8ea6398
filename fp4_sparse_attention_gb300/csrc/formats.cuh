// formats.cuh -- the two block-scaled FP4 formats as the tensor core sees them.
//
// Both store E2M1 codes, two per byte, 128 values (64 bytes) per row; they
// differ in the block scale (M3-indexer README, "FP4 和 scale layout"):
//   MXFP4: one E8M0 scale per 32 values (G = 4 per row), scale_vec::2X, ue8m0;
//          one 32x4x4 scale atom serves both K = 64 halves of a row (sf_id 0 / 2).
//   NVFP4: one E4M3 scale per 16 values (G = 8 per row), scale_vec::4X, ue4m3;
//          one atom per K = 64 half (scales 0..3 and 4..7).
#pragma once

namespace fp4idx {

template <int FMT>
struct FmtTraits;
template <>
struct FmtTraits<0> {  // MXFP4
  static constexpr int G = 4, kAtoms = 1, kScaleVec = 2;
  static constexpr bool kUe8m0 = true;
};
template <>
struct FmtTraits<1> {  // NVFP4
  static constexpr int G = 8, kAtoms = 2, kScaleVec = 4;
  static constexpr bool kUe8m0 = false;
};

}  // namespace fp4idx
