// kv_store.cu -- write new K/V rows into the paged cache through slot_mapping.
//
// The engine's attention layer stores each new token's key and value into the
// preallocated cache blocks at the slot its block manager chose (nano-vllm hub
// page, "core tech 2: Attention + Triton kernel"; fixed 256-token blocks,
// "core tech 4").  This is a pure bit copy, HBM bound: one warp moves one
// token, 16 bytes per lane per access, all loads of a lane issued before its
// stores.
#include "host_common.h"
#include "pkv_common.cuh"

namespace pkv {
namespace {

constexpr int kWarpsPerCta = 8;

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// row_vecs: 16-byte vectors per row (Hkv*D/8).  Strides in vectors.
template <int kUnroll>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    kv_store_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                    uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                    const int32_t *__restrict__ slot_mapping, int64_t num_tokens, int row_vecs,
                    int64_t k_stride, int64_t v_stride, int64_t num_slots, int32_t *status) {
  const int64_t t = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= num_tokens) return;
  const int64_t slot = __ldg(slot_mapping + t);
  if (slot < 0 || slot >= num_slots) {
    if (slot != -1 && lane == 0) flag_status(status, PKV_DEV_BAD_SLOT);
    return;
  }
  const uint4 *ks = k + t * k_stride;
  const uint4 *vs = v + t * v_stride;
  uint4 *kd = k_cache + slot * row_vecs;
  uint4 *vd = v_cache + slot * row_vecs;
  for (int base = 0; base < row_vecs; base += 32 * kUnroll) {
    uint4 a[kUnroll], b[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * 32 + lane;
      if (i < row_vecs) {
        a[u] = ld_stream(ks + i);
        b[u] = ld_stream(vs + i);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * 32 + lane;
      if (i < row_vecs) {
        kd[i] = a[u];
        vd[i] = b[u];
      }
    }
  }
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_kv_store(const uint16_t *k, const uint16_t *v, uint16_t *k_cache,
                                   uint16_t *v_cache, const int32_t *slot_mapping,
                                   int64_t num_tokens, int num_kv_heads, int head_dim,
                                   int64_t k_token_stride, int64_t v_token_stride,
                                   int64_t num_blocks, int block_size, int32_t *dev_status,
                                   void *stream) {
  using namespace pkv;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 ||
      block_size <= 0)
    return PKV_ERR_INVALID_ARG;
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  if (row % 8 != 0) return PKV_ERR_UNSUPPORTED;
  if (k_token_stride == 0) k_token_stride = row;
  if (v_token_stride == 0) v_token_stride = row;
  if (k_token_stride < row || v_token_stride < row || k_token_stride % 8 != 0 ||
      v_token_stride % 8 != 0)
    return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  const int row_vecs = (int)(row / 8);
  const int64_t blocks = (num_tokens + kWarpsPerCta - 1) / kWarpsPerCta;
  if (blocks > 0x7FFFFFFFLL) return PKV_ERR_INVALID_ARG;
  kv_store_kernel<4><<<(unsigned)blocks, kWarpsPerCta * 32, 0, (cudaStream_t)stream>>>(
      reinterpret_cast<const uint4 *>(k), reinterpret_cast<const uint4 *>(v),
      reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache), slot_mapping,
      num_tokens, row_vecs, k_token_stride / 8, v_token_stride / 8,
      num_blocks * (int64_t)block_size, dev_status);
  return launch_status();
}
