// dequant.cu -- W4A16-G128 weight dequantisation: int32-packed 4-bit -> bf16.
//
// A quantised weight is an int32 tensor in which each int32 packs eight 4-bit
// values; dequantisation is int32 -> u4 unpack -> s4 reconstruct -> float x
// weight_scale, one scale per group of 128 weights (s1nh.org post on
// upgrading nano-vllm to big-vLLM, section on quantisation).  Layout read
// here: nibble i of a word is bits 4i..4i+3, s4 = u4 - 8, W [N, K] with
// packed [N, K/8], scales [N, K/128] bf16, out [N, K] bf16.
//
// Design (GB300): HBM-bound streaming, 16 bytes in and 64 bytes out per 32
// weights.  A persistent grid (SMs x 8 CTAs of 256 threads) walks 32-weight
// chunks, four per thread per pass with their loads issued first: per chunk
// one 16-byte streaming load of four words, one scale, 32 products
// in bf16 pairs (u - 8 is exact in bf16; the multiply rounds the exact
// product once to nearest even, as rounding an fp32 product would: that
// product needs at most 12 significant bits), and two 32-byte (or four
// 16-byte) stores.
#include "host_common.h"
#include "pkv_common.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 8;

__device__ __forceinline__ uint4 ld_stream_u4(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_v8(void *p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Eight weights of one word, as four packed bf16 pairs (lower index in the
// low half).  (word >> 4j) & 0x000F000F | 0x43004300 is the bf16 pair
// (128 + u_j, 128 + u_{j+4}) exactly (bf16 holds every integer up to 256);
// subtracting the pair (136, 136) gives (u - 8) exactly, and one bf16x2
// multiply by the scale rounds the exact product once to nearest even.
// Byte permutes then put the pairs in element order (0,1) (2,3) (4,5) (6,7).
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ void dequant_word(uint32_t word, uint32_t scale2, uint32_t *out4) {
  constexpr uint32_t kBias = 0x43084308u;  // bf16 pair (136, 136)
  uint32_t r[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t x = ((word >> (4 * j)) & 0x000F000Fu) | 0x43004300u;  // (128+u_j, 128+u_{j+4})
    r[j] = bf16x2_mul(bf16x2_sub(x, kBias), scale2);
  }
  out4[0] = prmt(r[0], r[1], 0x5410u);  // (w0, w1)
  out4[1] = prmt(r[2], r[3], 0x5410u);  // (w2, w3)
  out4[2] = prmt(r[0], r[1], 0x7632u);  // (w4, w5)
  out4[3] = prmt(r[2], r[3], 0x7632u);  // (w6, w7)
}

// U chunks per thread per pass, their loads issued before any arithmetic so
// that more bytes are in flight per thread; I is the index type (32-bit when
// every chunk index fits, which saves integer work per chunk).
template <int U, typename I>
__global__ void __launch_bounds__(kThreads)
    w4a16_dequant_kernel(uint16_t *__restrict__ out, const int32_t *__restrict__ packed,
                         const uint16_t *__restrict__ scales, int64_t chunks_,
                         int64_t chunks_per_row_, int64_t groups_per_row_, int out_32b) {
  const I chunks = (I)chunks_, cpr = (I)chunks_per_row_, gpr = (I)groups_per_row_;
  const I stride = (I)gridDim.x * kThreads;
  for (I c0 = (I)blockIdx.x * kThreads + threadIdx.x; c0 < chunks; c0 += stride * U) {
    uint4 w[U];
    uint32_t sc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const I c = c0 + (I)u * stride;
      if (c < chunks) {
        const I row = c / cpr;  // chunk in row: c - row * cpr, 32 weights each
        w[u] = ld_stream_u4(packed + (int64_t)c * 4);
        sc[u] = __ldg(scales + (int64_t)row * gpr + (c - row * cpr) / 4);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const I c = c0 + (I)u * stride;
      if (c < chunks) {
        const uint32_t scale = sc[u] | (sc[u] << 16);  // the scale in both halves
        uint32_t o[16];
        dequant_word(w[u].x, scale, o);
        dequant_word(w[u].y, scale, o + 4);
        dequant_word(w[u].z, scale, o + 8);
        dequant_word(w[u].w, scale, o + 12);
        uint16_t *dst = out + (int64_t)c * 32;
        if (out_32b) {
          st_v8(dst, *reinterpret_cast<const uint32_t(*)[8]>(o));
          st_v8(dst + 16, *reinterpret_cast<const uint32_t(*)[8]>(o + 8));
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            reinterpret_cast<uint4 *>(dst)[q] =
                make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        }
      }
    }
  }
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_w4a16_dequant(uint16_t *out, const int32_t *packed,
                                        const uint16_t *scales, int64_t n_rows, int64_t k,
                                        int group_size, void *stream) {
  using namespace pkv;
  if (n_rows < 0 || k < 0) return PKV_ERR_INVALID_ARG;
  if (group_size != 128) return PKV_ERR_UNSUPPORTED;
  if (k % 128 != 0) return PKV_ERR_INVALID_ARG;
  if (n_rows == 0 || k == 0) return PKV_OK;
  if (!out || !packed || !scales) return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(packed) || (reinterpret_cast<uintptr_t>(scales) & 1u) != 0)
    return PKV_ERR_INVALID_ARG;
  const int64_t chunks_per_row = k / 32;
  if (n_rows > INT64_MAX / chunks_per_row) return PKV_ERR_INVALID_ARG;
  const int64_t chunks = n_rows * chunks_per_row;
  int64_t grid = (int64_t)device_sm_count() * kCtasPerSm;
  const int64_t need = (chunks + kThreads - 1) / kThreads;
  if (grid > need) grid = need;
  const int out_32b = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0;
  constexpr int U = 4;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // 32-bit indices when no chunk index (plus a pass's stride) can overflow them.
  if (chunks + grid * kThreads * U < ((int64_t)1 << 32))
    w4a16_dequant_kernel<U, uint32_t><<<(unsigned)grid, kThreads, 0, st>>>(
        out, packed, scales, chunks, chunks_per_row, k / 128, out_32b);
  else
    w4a16_dequant_kernel<U, int64_t><<<(unsigned)grid, kThreads, 0, st>>>(
        out, packed, scales, chunks, chunks_per_row, k / 128, out_32b);
  return launch_status();
}
