// store_k.cu -- MXFP4 K-cache writer: bf16 keys -> E2M1 codes + E8M0 scales
// in the paged cache layout (SGLang PR 42861: store_fp4_index_k_cache with
// round-to-nearest-even; E8M0 exponents clamped to 1..254).  With no slot
// table (slots == nullptr) token i goes to slot i; on one-token pages that
// is the dense query layout [T][H][64] / [T][H][4], which is how bf16
// queries are quantised (fp4idx_quantize_q).
//
// One thread per 32-value group of one (token, K head) row: four 16-byte
// loads of bf16, the group's max magnitude, the shared exponent from its
// float exponent field, then each value placed on the E2M1 grid by
// comparisons against the midpoints between levels (a tie goes to the level
// with the even index, i.e. the even mantissa), 16 bytes of codes and one
// scale byte stored.  Memory-bound: 64 bytes read, 17 written per group.
#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace fp4idx {
namespace {

constexpr int kStoreThreads = 256;

// E2M1 index (0..7) of |y| rounded to the nearest level of
// [0, 0.5, 1, 1.5, 2, 3, 4, 6], ties to the even index, saturating at 6.
__device__ __forceinline__ uint32_t e2m1_rne_index(float a) {
  uint32_t i = 0;
  i += a > 0.25f;
  i += a >= 0.75f;  // tie 0.75 -> 1.0 (index 2)
  i += a > 1.25f;
  i += a >= 1.75f;  // tie 1.75 -> 2.0 (index 4)
  i += a > 2.5f;
  i += a >= 3.5f;   // tie 3.5 -> 4.0 (index 6)
  i += a > 5.0f;
  return i;
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
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
  // floor(log2(amax)) of a normal float is its exponent field - 127; the
  // E2M1 largest exponent is 2, so code = field - 2, clamped (a zero or
  // subnormal max gives code 1)
  const int field = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF);
  const int code = field - 2 < 1 ? 1 : (field - 2 > 254 ? 254 : field - 2);
  // 1 / scale = 2^(127 - code), exact: exponent field 254 - code (code 254,
  // unreachable from a finite max, would be the subnormal 2^-127)
  const float inv = code <= 253 ? __uint_as_float(static_cast<uint32_t>(254 - code) << 23) : 0x1p-127f;
  uint32_t packed[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float y = x[i] * inv;
    const uint32_t idx = e2m1_rne_index(fabsf(y));
    const uint32_t nib = idx | ((idx != 0 && (__float_as_uint(x[i]) >> 31)) ? 8u : 0u);
    packed[i >> 3] |= nib << (4 * (i & 7));
  }
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
