// store_k.cu -- MXFP4 K-cache writer: bf16 keys -> E2M1 codes + E8M0 scales
// in the paged cache layout (SGLang PR 42861: store_fp4_index_k_cache with
// round-to-nearest-even; E8M0 exponents clamped to 1..254).  With no slot
// table (slots == nullptr) token i goes to slot i; on one-token pages that
// is the dense query layout [T][H][64] / [T][H][4], which is how bf16
// queries are quantised (fp4idx_quantize_q).
//
// One thread per 32-value group of one (token, K head) row: four 16-byte
// loads of bf16, the group's max magnitude, the shared exponent from its
// float exponent field, then each scaled value converted to E2M1 by the
// hardware conversion (round to nearest, ties to the even mantissa, i.e. the
// level with the even index; saturating at 6), 16 bytes of codes and one
// scale byte stored.  A value that rounds to zero is stored as +0, and a NaN
// value as +0 (a group holding one takes a slower path that also leaves it
// out of the max).  Memory-bound: 64 bytes read, 17 written per group.
#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace fp4idx {
namespace {

constexpr int kStoreThreads = 256;

// Eight values to eight E2M1 codes (value j in bits 4j..4j+3): round to
// the nearest of [0, 0.5, 1, 1.5, 2, 3, 4, 6] with ties to the even
// mantissa, saturating, sign in bit 3 -- then a zero magnitude loses its
// sign, so every value that rounds to zero is stored as +0.
__device__ __forceinline__ uint32_t e2m1x8(const float* y) {
  uint32_t w;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(w)
      : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]), "f"(y[6]), "f"(y[7]));
  const uint32_t nz = (w | (w >> 1) | (w >> 2)) & 0x11111111u;  // bit 0 of a nibble: magnitude != 0
  return w & (0x77777777u | (nz << 3));
}

__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

__global__ void __launch_bounds__(kStoreThreads) store_k_kernel(const StoreParams p) {
  pdl_wait();  // the keys may come from the kernel before this one
  pdl_launch_dependents();
  const int64_t gidx = static_cast<int64_t>(blockIdx.x) * kStoreThreads + threadIdx.x;
  const int64_t groups = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads * 4;
  if (gidx >= groups) return;
  const int g = static_cast<int>(gidx & 3);
  const int64_t row = gidx >> 2;  // token * Hkv + head
  const int64_t tok = row / p.num_kv_heads;
  const int hk = static_cast<int>(row - tok * p.num_kv_heads);
  const int64_t slot = p.slots ? static_cast<int64_t>(__ldg(p.slots + tok)) : tok;
  if (slot < 0) return;
  if (slot >= p.num_pages * p.page_size) {
    if (g == 0 && hk == 0) atomicOr(p.err, kErrPageRange);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(p.keys + tok * p.key_row_stride + hk * 128 + g * 32);
  uint32_t w[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 v = __ldg(src + q);
    w[4 * q] = v.x;
    w[4 * q + 1] = v.y;
    w[4 * q + 2] = v.z;
    w[4 * q + 3] = v.w;
  }
  // bf16 -> fp32 is exact (the 16 bits become the high half)
  float x[32];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = max_nan(amax, fabsf(x[i]));
  if (isnan(amax)) {  // NaN values: left out of the max, stored as +0
    amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      x[i] = isnan(x[i]) ? 0.0f : x[i];
      amax = fmaxf(amax, fabsf(x[i]));
    }
  }
  // floor(log2(amax)) of a normal float is its exponent field - 127; the
  // E2M1 largest exponent is 2, so code = field - 2, clamped (a zero or
  // subnormal max gives code 1)
  const int field = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF);
  const int code = field - 2 < 1 ? 1 : (field - 2 > 254 ? 254 : field - 2);
  // 1 / scale = 2^(127 - code), exact: exponent field 254 - code (code 254,
  // unreachable from a finite max, would be the subnormal 2^-127)
  const float inv = code <= 253 ? __uint_as_float(static_cast<uint32_t>(254 - code) << 23) : 0x1p-127f;
  // x * inv is exact (a power-of-two scale of a bf16 value)
  float y[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) y[i] = x[i] * inv;
  uint32_t packed[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) packed[q] = e2m1x8(y + 8 * q);
  const int64_t blk = static_cast<int64_t>(slot / p.page_size) * p.num_kv_heads + hk;  // (page, K head)
  const int64_t off = slot % p.page_size;
  uint8_t* codes;
  uint8_t* scales;
  if (p.fused) {  // [page*64 code bytes][page*4 scale bytes] per block
    codes = p.k + blk * p.page_size * 68 + off * 64;
    scales = p.k + blk * p.page_size * 68 + static_cast<int64_t>(p.page_size) * 64 + off * 4;
  } else {
    codes = p.k + (blk * p.page_size + off) * 64;
    scales = p.k_scale + (blk * p.page_size + off) * 4;
  }
  *reinterpret_cast<uint4*>(codes + g * 16) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  scales[g] = static_cast<uint8_t>(code);
}

}  // namespace

cudaError_t launch_store_k(const StoreParams& p, cudaStream_t stream) {
  const int64_t groups = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads * 4;
  if (groups == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>((groups + kStoreThreads - 1) / kStoreThreads);
  // programmatic dependent launch: the next kernel may be scheduled while
  // this one runs (it waits for this one's writes with griddepcontrol.wait)
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kStoreThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, store_k_kernel, p);
}

}  // namespace fp4idx
