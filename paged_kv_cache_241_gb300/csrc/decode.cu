// decode.cu -- paged decode attention: split-K flash-decoding over a block table.
//
// Decode attends one new query token per sequence to the whole paged context;
// each step re-reads the sequence's cached keys and values, so it is bound by
// memory bandwidth (CSDN essay "from nanoVLLM to vLLM", Mountain 3 and the
// study route's note on the attention/ module).  The context lives in fixed
// 256-token blocks reached through the block table (same essay, Mountain 1;
// nano-vllm hub page, "core tech 4").
//
// Design (GB300):
//  * Work item = (sequence, kv head, logical block).  A persistent grid of
//    (#SM x resident CTAs) walks the items with no host sync: every CTA
//    derives the item list from context_lens itself (block-wide scan in
//    smem).  With many items per CTA they are handed out by an atomic counter
//    in the caller's workspace, each CTA taking the next one when its producer
//    is ready for it, so the CTAs finish together although items and SMs
//    differ in speed; with few, round-robin (the counter's round trip then
//    costs more than the balance gains).  The last CTA to finish leaves the
//    counter zeroed for the next call.  When there are very many items (24
//    or more per CTA, long contexts) and the host launches the kernel's
//    two-block form, an item spans two consecutive blocks of its sequence:
//    half the partials to write and merge and half the per-item costs (long
//    skewed decode 354.6 -> 347.1 us); the consumers carry the running max,
//    sum and unnormalised O from one block to the next.
//  * One producer warp streams each block's K tiles, then its V tiles, as 4-D
//    TMA boxes {D, 1 head, 64 tokens, 1 block} into a ring of shared-memory
//    stages; the block-table lookup is the box's outer coordinate.  With a
//    4-deep ring every other slot is filled instead by cp.async from the
//    warp's 32 lanes, a second load path beside the TMA unit.
//  * Four consumer warps compute in fp32 on the CUDA cores (decode is
//    HBM-bound: no GEMM reshaping).  All G = Hq/Hkv query heads of the group
//    share each K/V tile read.  Phase 1: logits for the item's tokens (lane
//    octets split D, a transposed shuffle reduction sums them).  Phase 2: exact
//    softmax statistics of the item.  Phase 3: P.V with each lane owning D/32
//    output dims.
//  * Each item writes a partial (max, sum, unnormalised output) to the
//    workspace; a merge kernel, launched as a programmatic dependent of this
//    grid (it waits for the grid's completion), combines each multi-item
//    (sequence, kv head)'s partials in parallel and writes bf16.  A sequence
//    that fits one item skips the workspace.
#include <math.h>

#include <mutex>

#include "host_common.h"
#include "pkv_common.cuh"

namespace pkv {
namespace {

constexpr int kTile = 64;           // tokens per TMA tile
constexpr int kConsumerWarps = 4;   // compute warps per CTA
constexpr int kThreads = (kConsumerWarps + 1) * 32;
// Shared-memory tile ring depth: 4 stages, 3 for groups of 4+ query heads so
// that three CTAs still fit on an SM.
__host__ __device__ constexpr int decode_stages(int G) { return G >= 4 ? 3 : 4; }
constexpr int kMaxSeqs = 16384;
constexpr int kItemSlots = 4;       // depth of the shared ring of fetched item indices
// Items per CTA from which they are handed out by the counter instead of
// round-robin: measured, long skewed decode (33 per CTA) 365 -> 351 us with
// the counter, the 64-sequence decode batch (6 per CTA) 60.1 -> 61.2 us.
constexpr int kCounterRounds = 12;
// Items per CTA (of one block each) from which an item spans two blocks of
// its sequence: half the partials to write and merge, half the per-item costs.
constexpr int kSpanRounds = 24;

// Test-only fault injection, set by pkv_test_decode_fault: the producer of
// every CTA skips the tile it would issue as its number `withhold` (counting
// from 0; -1 = none), so that tile's consumers wait until the wait limit runs
// out.  Read once per CTA.
static __device__ int g_decode_withhold_tile = -1;
constexpr int kMaxDynamicSmem = 232448;  // opt-in shared memory per CTA on sm_103 (227 KiB)
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
  uint16_t *out;
  unsigned int *ctl;    // [0]: next item to hand out, [1]: CTAs done (both 0 between calls)
  const uint16_t *q;
  const int32_t *block_tables;
  const int32_t *context_lens;
  int32_t *seq_prefix;  // [num_seqs + 1]: first partial (block) index of each sequence
  float *part_ml;     // [max_total_blocks, Hq, 2]   (max in log2 units, sum)
  float *part_o;      // [max_total_blocks, Hq, D]
  int32_t *status;
  int64_t num_blocks;
  int64_t max_total_blocks;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int block_size;
  int max_blocks_per_seq;
  float qscale;  // scale * log2(e)
  // Two-block form only: items may span two blocks (the host sets it when it
  // launches that form; a run-time flag rather than a constant because ptxas
  // then allocates the form's registers without a spill).
  int span_ok;
  // Fused store (all null unless the call also stores this step's tokens):
  // row s of new_k / new_v is the token at position context_lens[s] - 1 of
  // sequence s, to be written to cache slot new_slots[s].
  const uint16_t *new_k;
  const uint16_t *new_v;
  const int32_t *new_slots;
  uint16_t *k_cache_w;
  uint16_t *v_cache_w;
  // The caches again, for the tiles the producer warp copies with cp.async.
  const uint16_t *k_cache_r;
  const uint16_t *v_cache_r;
};

// With a 4-deep ring, the odd slots are filled by cp.async from all 32 lanes
// of the producer warp (each lane's copies complete with an arrive on the
// slot's barrier), the others by TMA from lane 0.  TMA alone lands ~5.7 TB/s
// over the GPU on this access pattern, TMA and the load/store path together
// ~6.4 TB/s (measured, K/V tiles streamed from HBM).  A 3-deep ring (groups of
// 4+ query heads) keeps TMA only: there the extra producer lanes cost the
// consumer warps more than the second path gains (measured).
template <int NS>
__host__ __device__ constexpr bool slot_by_lanes(int st) { return NS % 2 == 0 && (st & 1) != 0; }

__device__ __forceinline__ void cp_async16_hint(uint32_t dst, const void *src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst),
               "l"(src), "l"(policy)
               : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the barrier counts this arrival among its expected ones).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ int named_bar_or(int id, int nthreads, int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %3, 0;\n\t"
      "bar.red.or.pred q, %1, %2, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(id), "r"(nthreads), "r"(pred)
      : "memory");
  return r;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Blocks held by a sequence of context length L (clamped; *bad set on a bad L).
__device__ __forceinline__ int seq_blocks(int L, int bs, int max_blocks, int *bad) {
  if (L <= 0) {
    *bad = 1;
    return 0;
  }
  int nb = (L + bs - 1) / bs;
  if (nb > max_blocks) {
    *bad = 1;
    nb = max_blocks;
  }
  return nb;
}

// Sum NV partial values over the 8 lanes of a lane octet (lane bits 0..2).
// Transposed reduction: every xor step halves the live values.  Afterwards
// lane r holds max(NV/8, 1) complete sums in v[0..): the values with original
// index octet_base<NV>(r) + u.  For NV == 4, lanes r and r^1 hold the same sum.
template <int NV>
__device__ __forceinline__ void octet_reduce(float (&v)[NV], int r) {
  static_assert(NV >= 4 && (NV & (NV - 1)) == 0, "NV must be a power of two >= 4");
  constexpr int H1 = NV / 2;
  {
    const bool hi = (r & 4) != 0;
#pragma unroll
    for (int u = 0; u < H1; ++u) {
      const float send = hi ? v[u] : v[u + H1];
      const float keep = hi ? v[u + H1] : v[u];
      v[u] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
  }
  constexpr int H2 = H1 / 2;
  {
    const bool hi = (r & 2) != 0;
#pragma unroll
    for (int u = 0; u < H2; ++u) {
      const float send = hi ? v[u] : v[u + H2];
      const float keep = hi ? v[u + H2] : v[u];
      v[u] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
  }
  if constexpr (H2 >= 2) {
    constexpr int H3 = H2 / 2;
    const bool hi = (r & 1) != 0;
#pragma unroll
    for (int u = 0; u < H3; ++u) {
      const float send = hi ? v[u] : v[u + H3];
      const float keep = hi ? v[u + H3] : v[u];
      v[u] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
    }
  } else {
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
  }
}

template <int NV>
__device__ __forceinline__ int octet_base(int r) {
  if constexpr (NV >= 8) {
    return ((r & 4) ? NV / 2 : 0) + ((r & 2) ? NV / 4 : 0) + ((r & 1) ? NV / 8 : 0);
  } else {
    return ((r & 4) ? 2 : 0) + ((r & 2) ? 1 : 0);
  }
}

// The G probability pairs of one token (16-byte vector loads where possible).
template <int G>
__device__ __forceinline__ void load_prob_pairs(const float2 *p, float2 (&pv)[G]) {
  if constexpr (G == 1) {
    pv[0] = p[0];
  } else {
#pragma unroll
    for (int i = 0; i < G; i += 2) {
      const float4 a = *reinterpret_cast<const float4 *>(p + i);
      pv[i] = make_float2(a.x, a.y);
      pv[i + 1] = make_float2(a.z, a.w);
    }
  }
}

// Shared-memory carve-up (bytes), shared by host and device.
struct DecodeSmem {
  int tiles, qbuf, bars, logits, red, stats, misc, iring, prefix, ctx, total;
  __host__ __device__ DecodeSmem(int D, int G, int bs, int num_seqs) {
    tiles = 0;
    const int stages = decode_stages(G);
    qbuf = tiles + stages * kTile * D * 2;  // [2][G*D] bf16: q of the next items
    // full[S], empty[S], q_full[2], q_empty[2], item_full[R], item_empty[R]
    bars = qbuf + 2 * G * D * 2;
    logits = bars + (2 * stages + 4 + 2 * kItemSlots) * 8;  // [block_size][G] float pairs
    red = logits + ((bs * G * 8 + 15) & ~15);
    stats = red + kConsumerWarps * G * D * 4;
    misc = stats + 3 * G * 4;
    iring = misc + 16;                      // [R] fetched item indices
    prefix = iring + kItemSlots * 4;
    ctx = prefix + (num_seqs + 1) * 4;
    total = ctx + num_seqs * 4;
  }
};

// 1-D bulk copy global -> shared, completing on an mbarrier (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

template <int D, int G, bool kSpan>
__global__ void __launch_bounds__(kThreads, G < 8 ? 3 : 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  constexpr int kStages = decode_stages(G);
  constexpr int kTileBytes = kTile * D * 2;
  constexpr int kQBytes = G * D * 2;
  constexpr int CPL = D / 64;  // 16-byte chunks per lane per token (phase 1)
  constexpr int DPL = D / 32;  // output dims per lane (phase 3)
  constexpr int NV = 4 * G;    // partial dot products per lane (phase 1)

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const DecodeSmem lay(D, G, p.block_size, p.num_seqs);
  uint8_t *tiles = smem + lay.tiles;
  uint8_t *qbuf = smem + lay.qbuf;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bars);
  uint64_t *empty = full + kStages;
  uint64_t *q_full = empty + kStages;
  uint64_t *q_empty = q_full + 2;
  uint64_t *item_full = q_empty + 2;        // [kItemSlots]: an item index is in the ring
  uint64_t *item_empty = item_full + kItemSlots;
  volatile int *iring = reinterpret_cast<volatile int *>(smem + lay.iring);
  // Per token and head: phase 1 stores the logit in .x, phase 2 replaces the
  // pair by (p, p) so phase 3 can feed it straight to a packed FMA.
  float2 *logits = reinterpret_cast<float2 *>(smem + lay.logits);  // [block_size][G]
  float *red = reinterpret_cast<float *>(smem + lay.red);        // [warps][G][D]
  float *mstat = reinterpret_cast<float *>(smem + lay.stats);    // [G]
  float *lstat = mstat + G;                                      // [G]
  float *astat = lstat + G;  // [G]: factor for what earlier blocks of the item left in O
  int *misc = reinterpret_cast<int *>(smem + lay.misc);          // abort flag
  int *prefix = reinterpret_cast<int *>(smem + lay.prefix);      // [num_seqs + 1]
  int *ctx = reinterpret_cast<int *>(smem + lay.ctx);            // [num_seqs], clamped
  volatile int *abort_flag = misc;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int S = p.num_seqs;
  const int BS = p.block_size;
  const int Hkv = p.num_kv_heads;
  const int Hq = p.num_q_heads;
  const int max_ctx = p.max_blocks_per_seq * BS;

  // ---- prologue: barriers, clamped lengths and the block prefix -----------
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], slot_by_lanes<kStages>(i) ? 32 : 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], kConsumerWarps);
    }
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], kConsumerWarps);
    }
    misc[0] = 0;
    fence_barrier_init();
  }
  if (tid == kConsumerWarps * 32) {
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
  }
  const int per = (S + kThreads - 1) / kThreads;
  const int s_begin = min(tid * per, S);
  const int s_end = min(s_begin + per, S);
  int bad = 0;
  int local = 0;
  for (int s = s_begin; s < s_end; ++s) {
    const int L = p.context_lens[s];
    ctx[s] = L <= 0 ? 0 : min(L, max_ctx);
    local += seq_blocks(L, BS, p.max_blocks_per_seq, &bad);
  }
  if (bad && blockIdx.x == 0) flag_status(p.status, PKV_DEV_BAD_CONTEXT);
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  // Warp totals go to the (still unused) reduction area.
  if (lane == 31) red[warp] = __int_as_float(incl);
  __syncthreads();
  int offset = incl - local;
  int total = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    const int wt = __float_as_int(red[w]);
    if (w < warp) offset += wt;
    total += wt;
  }
  {
    int run = offset;
    for (int s = s_begin; s < s_end; ++s) {
      prefix[s] = run;
      run += (ctx[s] + BS - 1) / BS;
    }
    if (tid == 0) prefix[S] = total;
  }
  __syncthreads();
  // Block 0 publishes the prefix for the merge kernel (all zeros, i.e. nothing
  // to merge, when the workspace bound is exceeded).
  const bool overflow = (int64_t)total > p.max_total_blocks;
  if (overflow) {
    if (blockIdx.x == 0)
      for (int i = tid; i <= S; i += kThreads) p.seq_prefix[i] = 0;
    if (blockIdx.x == 0 && tid == 0) flag_status(p.status, PKV_DEV_WORKSPACE);
    return;
  }
  // With many items per CTA an item spans two blocks: the prefix then counts
  // items of each sequence (its partials), ceil(blocks / 2).
  const int span = (kSpan && p.span_ok && total * Hkv >= kSpanRounds * (int)gridDim.x) ? 2 : 1;
  int total_parts = total;
  if (span == 2) {
    int lp = 0;
    for (int s = s_begin; s < s_end; ++s) lp += ((ctx[s] + BS - 1) / BS + 1) >> 1;
    int ip = lp;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, ip, o);
      if (lane >= o) ip += y;
    }
    if (lane == 31) red[warp] = __int_as_float(ip);
    __syncthreads();
    int off2 = ip - lp;
    int tot2 = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      const int wt = __float_as_int(red[w]);
      if (w < warp) off2 += wt;
      tot2 += wt;
    }
    int run = off2;
    for (int s = s_begin; s < s_end; ++s) {
      prefix[s] = run;
      run += ((ctx[s] + BS - 1) / BS + 1) >> 1;
    }
    if (tid == 0) prefix[S] = tot2;
    total_parts = tot2;
    __syncthreads();
  }
  if (blockIdx.x == 0)
    for (int i = tid; i <= S; i += kThreads) p.seq_prefix[i] = prefix[i];
  const int total_items = total_parts * Hkv;
  // The merge kernel may start launching now; it waits for this grid to finish.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // Item w: sequence s, kv head j, its first block b and its blocks nbi
  // (one, or two when items span two blocks), and its partial's index gblk.
  auto item_coords = [&](int w, int &s, int &b, int &nbi, int &j, int &gblk) {
    gblk = w / Hkv;
    j = w - gblk * Hkv;
    int lo = 0, hi = S - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= gblk)
        lo = mid;
      else
        hi = mid - 1;
    }
    s = lo;
    b = (gblk - prefix[s]) * span;
    nbi = kSpan ? min(span, (ctx[s] + BS - 1) / BS - b) : 1;
  };

  // Producer side of the item ring (lane 0 of the producer warp): the next
  // item index (from the shared counter, or round-robin), and its hand-over
  // to the consumers (an index >= total_items tells them to stop).
  const bool by_counter = total_items >= kCounterRounds * (int)gridDim.x;
  int round_no = 0;
  auto fetch_item = [&]() -> int {
    if (!by_counter) return (int)blockIdx.x + (round_no++) * (int)gridDim.x;
    return (int)atomicAdd(&p.ctl[0], 1u);
  };
  auto publish_item = [&](int item_no, int w) -> bool {
    const int slot = item_no % kItemSlots;
    if (item_no >= kItemSlots &&
        !mbar_wait_bounded(&item_empty[slot], ((item_no / kItemSlots) - 1) & 1, abort_flag))
      return false;
    iring[slot] = w;
    mbar_arrive(&item_full[slot]);  // (release: orders the store above)
    return true;
  };
  // Every CTA's producer calls this once on its way out: the last one resets
  // the counters for the next call on this workspace.
  auto leave = [&]() {
    __threadfence();
    if (atomicAdd(&p.ctl[1], 1u) == gridDim.x - 1) {
      p.ctl[0] = 0;
      p.ctl[1] = 0;
      __threadfence();
    }
  };

  // ---- producer warp: q, then K tiles, then V tiles of every item ----------
  // 3-deep ring: lane 0 alone issues the q copy and every tile by TMA.
  if (!slot_by_lanes<kStages>(1) && warp == kConsumerWarps) {
    if (lane == 0) {
      const int withhold = g_decode_withhold_tile;
      const uint64_t policy = l2_policy_evict_first();
      int issued = 0;
      int item_no = 0;
      bool ok = true;
      int s, b, nbi, j, gblk;
      int w = fetch_item();
      int blk_next = 0;
      if (w < total_items) {
        item_coords(w, s, b, nbi, j, gblk);
        blk_next = p.block_tables[(int64_t)s * p.max_blocks_per_seq + b];
      }
      for (;; ++item_no) {
        if (!publish_item(item_no, w)) {
          ok = false;
          break;
        }
        if (w >= total_items) break;
        const int wn = fetch_item();  // the next item (its value is first needed below)
        item_coords(w, s, b, nbi, j, gblk);
        const int qb = item_no & 1;
        if (item_no >= 2 &&
            !mbar_wait_bounded(&q_empty[qb], ((item_no >> 1) - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&q_full[qb], kQBytes);
        bulk_load(qbuf + qb * kQBytes, p.q + ((int64_t)s * Hq + j * G) * D, kQBytes,
                  &q_full[qb]);
        for (int bi = 0; bi < nbi && ok; ++bi) {
        int blk = bi == 0 ? blk_next : p.block_tables[(int64_t)s * p.max_blocks_per_seq + b + bi];
        if (blk < 0 || (int64_t)blk >= p.num_blocks) {
          flag_status(p.status, PKV_DEV_BAD_BLOCK);
          blk = 0;
        }
        const int valid = min(BS, ctx[s] - (b + bi) * BS);
        const int ntile = (valid + kTile - 1) / kTile;
        for (int half = 0; half < 2 && ok; ++half) {
          const CUtensorMap *map = half ? &tm_v : &tm_k;
          for (int t = 0; t < ntile; ++t) {
            const int st = issued % kStages;
            if (issued >= kStages &&
                !mbar_wait_bounded(&empty[st], ((issued / kStages) - 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            if (issued != withhold) {
              mbar_arrive_expect_tx(&full[st], kTileBytes);
              tma_load_4d_hint(tiles + st * kTileBytes, map, &full[st], 0, j, t * kTile, blk,
                               policy);
            }
            ++issued;
          }
        }
        }
        if (!ok) {
          ++item_no;  // this item's q copy was issued: the drain below waits for it
          break;
        }
        w = wn;
        if (w < total_items) {  // the next item's block id, read early
          int sn, bn, nn, jn, gn;
          item_coords(w, sn, bn, nn, jn, gn);
          blk_next = p.block_tables[(int64_t)sn * p.max_blocks_per_seq + bn];
        }
      }
      if (!ok) flag_status(p.status, PKV_DEV_TIMEOUT);
      // Do not leave while copies into this CTA's shared memory are in flight.
      for (int i = max(0, issued - kStages); i < issued; ++i)
        if (!mbar_wait_bounded(&full[i % kStages], (i / kStages) & 1, nullptr)) flag_status(p.status, PKV_DEV_TIMEOUT);
      for (int i = max(0, item_no - 2); i < item_no; ++i)
        if (!mbar_wait_bounded(&q_full[i & 1], (i >> 1) & 1, nullptr)) flag_status(p.status, PKV_DEV_TIMEOUT);
      leave();
    }
    return;
  }

  // 4-deep ring: every lane runs the loop (they share the cp.async slots);
  // lane 0 alone issues the q copy and the TMA tiles.
  if (warp == kConsumerWarps) {
    constexpr int kChunks = D / 8;       // 16-byte chunks per token row
    constexpr int kRowsPer = 32 / kChunks;  // token rows per warp-wide copy
    const uint64_t policy = l2_policy_evict_first();
    const int withhold = g_decode_withhold_tile;
    const int part = lane % kChunks;
    const int row0 = lane / kChunks;
    int issued = 0;
    int item_no = 0;
    bool ok = true;
    int s, b, nbi, j, gblk;
    int blk_next = 0;
    int w = lane == 0 ? fetch_item() : 0;
    w = __shfl_sync(0xffffffffu, w, 0);
    if (w < total_items) {
      item_coords(w, s, b, nbi, j, gblk);
      blk_next = p.block_tables[(int64_t)s * p.max_blocks_per_seq + b];
    }
    for (;; ++item_no) {
      {
        const bool good = lane == 0 ? publish_item(item_no, w) : true;
        ok = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
      if (w >= total_items) break;
      const int wn_lane0 = lane == 0 ? fetch_item() : 0;  // the next item, first needed below
      item_coords(w, s, b, nbi, j, gblk);
      const int qb = item_no & 1;
      if (item_no >= 2) {
        const bool good =
            lane == 0 ? mbar_wait_bounded(&q_empty[qb], ((item_no >> 1) - 1) & 1, abort_flag) : true;
        ok = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&q_full[qb], kQBytes);
        bulk_load(qbuf + qb * kQBytes, p.q + ((int64_t)s * Hq + j * G) * D, kQBytes,
                  &q_full[qb]);
      }
      for (int bi = 0; bi < nbi && ok; ++bi) {
      int blk = bi == 0 ? blk_next : p.block_tables[(int64_t)s * p.max_blocks_per_seq + b + bi];
      if (blk < 0 || (int64_t)blk >= p.num_blocks) {
        if (lane == 0) flag_status(p.status, PKV_DEV_BAD_BLOCK);
        blk = 0;
      }
      const int valid = min(BS, ctx[s] - (b + bi) * BS);
      const int ntile = (valid + kTile - 1) / kTile;
      for (int half = 0; half < 2 && ok; ++half) {
        const CUtensorMap *map = half ? &tm_v : &tm_k;
        const uint16_t *cache = half ? p.v_cache_r : p.k_cache_r;
        for (int t = 0; t < ntile; ++t) {
          const int st = issued % kStages;
          if (issued >= kStages) {
            const bool good = lane == 0 ? mbar_wait_bounded(&empty[st], ((issued / kStages) - 1) & 1,
                                                            abort_flag)
                                        : true;
            ok = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
            if (!ok) break;
          }
          if (issued == withhold) {
            // (test-only: nothing issued, the slot's consumers time out)
          } else if (slot_by_lanes<kStages>(st)) {
            // Token rows t*64 .. t*64+63 of block blk, kv head j: row r is
            // (blk*BS + t*64 + r)*Hkv + j rows of D into the cache.
            const uint16_t *src =
                cache + (((int64_t)blk * BS + t * kTile + row0) * Hkv + j) * D + part * 8;
            const uint32_t dst = smem_u32(tiles + st * kTileBytes) + row0 * D * 2 + part * 16;
#pragma unroll 8
            for (int k = 0; k < kTile / kRowsPer; ++k)
              cp_async16_hint(dst + k * kRowsPer * D * 2,
                              src + (int64_t)k * kRowsPer * Hkv * D, policy);
            cp_async_arrive_noinc(&full[st]);
          } else if (lane == 0) {
            mbar_arrive_expect_tx(&full[st], kTileBytes);
            tma_load_4d_hint(tiles + st * kTileBytes, map, &full[st], 0, j, t * kTile, blk,
                             policy);
          }
          ++issued;
        }
      }
      }
      if (!ok) {
        ++item_no;  // this item's q copy was issued: the drain below waits for it
        break;
      }
      w = __shfl_sync(0xffffffffu, wn_lane0, 0);
      if (w < total_items) {  // the next item's block id, read early
        int sn, bn, nn, jn, gn;
        item_coords(w, sn, bn, nn, jn, gn);
        blk_next = p.block_tables[(int64_t)sn * p.max_blocks_per_seq + bn];
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (lane == 0) {
      if (!ok) flag_status(p.status, PKV_DEV_TIMEOUT);
      // Do not leave while copies into this CTA's shared memory are in flight.
      for (int i = max(0, issued - kStages); i < issued; ++i)
        if (!mbar_wait_bounded(&full[i % kStages], (i / kStages) & 1, nullptr))
          flag_status(p.status, PKV_DEV_TIMEOUT);
      for (int i = max(0, item_no - 2); i < item_no; ++i)
        if (!mbar_wait_bounded(&q_full[i & 1], (i >> 1) & 1, nullptr))
          flag_status(p.status, PKV_DEV_TIMEOUT);
      leave();
    }
    return;
  }

  // ---- consumer warps -----------------------------------------------------
  const int r = lane & 7;     // lane within its octet
  const int gid = lane >> 3;  // octet index: 4 tokens each
  int ctile = 0;              // tiles consumed so far
  for (int item_no = 0;; ++item_no) {
    // The next item index from the producer's ring; the four warps decide
    // together whether to go on (a wait that ran out stops all of them).
    int w = total_items;
    {
      const int slot = item_no % kItemSlots;
      const bool got =
          mbar_wait_bounded(&item_full[slot], (item_no / kItemSlots) & 1, abort_flag);
      if (got) w = iring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[slot]);
      if (named_bar_or(1, kConsumerWarps * 32, (!got || w >= total_items) ? 1 : 0)) {
        if (!got && tid == 0) flag_status(p.status, PKV_DEV_TIMEOUT);
        break;
      }
    }
    int s, b, nbi, j, gblk;
    item_coords(w, s, b, nbi, j, gblk);
    const int nblk = prefix[s + 1] - prefix[s];  // the sequence's items (partials)
    const int nb_seq = (ctx[s] + BS - 1) / BS;   // and its blocks
    const int h0 = j * G;

    // q of the item, staged by the producer (slot item_no & 1); read again
    // for each of the item's blocks and released after the last.
    const int qb = item_no & 1;
    const bool q_ok = mbar_wait_bounded(&q_full[qb], (item_no >> 1) & 1, abort_flag);
    const uint16_t *qs = reinterpret_cast<const uint16_t *>(qbuf + qb * kQBytes);

    // O accumulates over the item's blocks (unnormalised); between blocks
    // each warp keeps its share in its part of the reduction area.
    float2 acc_o[G][DPL / 2];
    for (int bi = 0; bi < nbi; ++bi) {
      const int bb = b + bi;
      const int valid = min(BS, ctx[s] - bb * BS);
      const int ntile = (valid + kTile - 1) / kTile;

      // q fragment: dim pairs (2e, 2e+1) of chunks r + 8c, in log2 units.
      float2 qf[G][CPL * 4];
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          uint4 raw = make_uint4(0, 0, 0, 0);
          if (q_ok) raw = *reinterpret_cast<const uint4 *>(qs + h * D + (r + 8 * c) * 8);
          const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            qf[h][c * 4 + e] = make_float2(bf16lo(wv[e]) * p.qscale, bf16hi(wv[e]) * p.qscale);
        }
      }
      if (bi == nbi - 1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_empty[qb]);
      }

      // Fused store: the item that holds the sequence's newest token takes that
      // token's K/V row from the inputs (patched into its shared-memory tiles,
      // so it never depends on the cache write) and stores it to the cache once
      // its tiles are consumed.  pl = the token's index inside this block.
      int pl = -1;
      uint4 new_krow = make_uint4(0, 0, 0, 0), new_vrow = make_uint4(0, 0, 0, 0);
      if (p.new_k != nullptr && bb == nb_seq - 1 && ctx[s] == p.context_lens[s]) {
        pl = ctx[s] - 1 - bb * BS;
        if (lane < D / 8) {
          const int64_t row = ((int64_t)s * Hkv + j) * D + lane * 8;
          new_krow = __ldg(reinterpret_cast<const uint4 *>(p.new_k + row));
          new_vrow = __ldg(reinterpret_cast<const uint4 *>(p.new_v + row));
        }
      }

      // Phase 1: logits of the item's tokens.
      for (int t = 0; t < ntile; ++t, ++ctile) {
        const int st = ctile % kStages;
        const bool ok = mbar_wait_bounded(&full[st], (ctile / kStages) & 1, abort_flag);
        if (ok) {
          const uint16_t *tile = reinterpret_cast<const uint16_t *>(tiles + st * kTileBytes);
          const int tok0 = warp * 16 + gid * 4;
          if (pl >= 0 && (pl >> 6) == t && warp == ((pl & 63) >> 4)) {
            if (lane < D / 8)
              reinterpret_cast<uint4 *>(tiles + st * kTileBytes + (pl & 63) * D * 2)[lane] = new_krow;
            __syncwarp();
          }
          // Packed FP32x2 FMAs: even and odd dims accumulate in the two halves.
          float2 acc2[NV];
#pragma unroll
          for (int i = 0; i < NV; ++i) acc2[i] = make_float2(0.f, 0.f);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint16_t *krow = tile + (tok0 + i) * D;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
              const uint4 raw = *reinterpret_cast<const uint4 *>(krow + (r + 8 * c) * 8);
              const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 kk = make_float2(bf16lo(wv[e]), bf16hi(wv[e]));
#pragma unroll
                for (int h = 0; h < G; ++h)
                  acc2[i * G + h] = __ffma2_rn(qf[h][c * 4 + e], kk, acc2[i * G + h]);
              }
            }
          }
          float acc[NV];
#pragma unroll
          for (int i = 0; i < NV; ++i) acc[i] = acc2[i].x + acc2[i].y;
          octet_reduce<NV>(acc, r);
          const int base = octet_base<NV>(r);
          constexpr int kOwned = NV >= 8 ? NV / 8 : 1;
          if (NV >= 8 || (r & 1) == 0) {
#pragma unroll
            for (int u = 0; u < kOwned; ++u) {
              const int vi = base + u;
              const int i = vi / G;
              const int h = vi - i * G;
              logits[(t * kTile + tok0 + i) * G + h].x = acc[u];
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      named_bar_sync(1, kConsumerWarps * 32);

      // Phase 2: softmax statistics of this block, per head, against the
      // running max of the item's blocks so far (log2 units); alpha rescales
      // what the earlier blocks left in O and l.
      for (int h = warp; h < G; h += kConsumerWarps) {
        float m = -INFINITY;
        for (int x = lane; x < valid; x += 32) m = fmaxf(m, logits[x * G + h].x);
        m = warp_max(m);
        const float m_old = bi == 0 ? -INFINITY : mstat[h];
        const float mn = fmaxf(m_old, m);
        float l = 0.f;
        for (int x = lane; x < valid; x += 32) {
          const float e = fast_exp2(logits[x * G + h].x - mn);
          logits[x * G + h] = make_float2(e, e);
          l += e;
        }
        l = warp_sum(l);
        if (lane == 0) {
          const float a = bi == 0 ? 0.f : fast_exp2(m_old - mn);
          mstat[h] = mn;
          lstat[h] = (bi == 0 ? 0.f : lstat[h] * a) + l;
          if constexpr (kSpan) astat[h] = a;
        }
      }
      named_bar_sync(1, kConsumerWarps * 32);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float a = kSpan ? astat[h] : 0.f;
#pragma unroll
        for (int e = 0; e < DPL / 2; ++e) {
          if (!kSpan || bi == 0) {
            acc_o[h][e] = make_float2(0.f, 0.f);
          } else {
            const float2 o =
                *reinterpret_cast<const float2 *>(red + (warp * G + h) * D + lane * DPL + 2 * e);
            acc_o[h][e] = make_float2(o.x * a, o.y * a);
          }
        }
      }

      // Phase 3: unnormalised P.V, lane owns dims [lane*DPL, lane*DPL + DPL).
      for (int t = 0; t < ntile; ++t, ++ctile) {
        const int st = ctile % kStages;
        const bool ok = mbar_wait_bounded(&full[st], (ctile / kStages) & 1, abort_flag);
        if (ok) {
          const uint16_t *tile = reinterpret_cast<const uint16_t *>(tiles + st * kTileBytes);
          const int tlo = warp * 16;
          if (pl >= 0 && (pl >> 6) == t && warp == ((pl & 63) >> 4)) {
            if (lane < D / 8)
              reinterpret_cast<uint4 *>(tiles + st * kTileBytes + (pl & 63) * D * 2)[lane] = new_vrow;
            __syncwarp();
          }
          const int thi = min(tlo + 16, valid - t * kTile);
#pragma unroll 4
          for (int tok = tlo; tok < thi; ++tok) {
            float2 vf[DPL / 2];
            if constexpr (DPL == 4) {
              const uint2 raw = *reinterpret_cast<const uint2 *>(tile + tok * D + lane * 4);
              vf[0] = make_float2(bf16lo(raw.x), bf16hi(raw.x));
              vf[1] = make_float2(bf16lo(raw.y), bf16hi(raw.y));
            } else {
              const uint32_t raw = *reinterpret_cast<const uint32_t *>(tile + tok * D + lane * 2);
              vf[0] = make_float2(bf16lo(raw), bf16hi(raw));
            }
            float2 pv[G];
            load_prob_pairs<G>(logits + (t * kTile + tok) * G, pv);
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
              for (int e = 0; e < DPL / 2; ++e) acc_o[h][e] = __ffma2_rn(pv[h], vf[e], acc_o[h][e]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }

      if (pl >= 0 && warp == 0) {
        const int64_t slot = p.new_slots[s];
        if (slot >= 0 && slot < p.num_blocks * BS) {
          if (lane < D / 8) {
            const int64_t row = (slot * Hkv + j) * D + lane * 8;
            *reinterpret_cast<uint4 *>(p.k_cache_w + row) = new_krow;
            *reinterpret_cast<uint4 *>(p.v_cache_w + row) = new_vrow;
          }
        } else if (slot != -1 && lane == 0) {
          flag_status(p.status, PKV_DEV_BAD_SLOT);
        }
      }

      if (bi + 1 < nbi) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < DPL / 2; ++e)
            *reinterpret_cast<float2 *>(red + (warp * G + h) * D + lane * DPL + 2 * e) =
                acc_o[h][e];
        // The next block's logits go where this block's probabilities are.
        named_bar_sync(1, kConsumerWarps * 32);
      }
    }

    // Epilogue: combine the four warps, then finish or publish a partial.
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < DPL / 2; ++e)
        *reinterpret_cast<float2 *>(red + (warp * G + h) * D + lane * DPL + 2 * e) = acc_o[h][e];
    named_bar_sync(1, kConsumerWarps * 32);
    if (nblk == 1) {
      for (int idx = tid; idx < G * D / 2; idx += kConsumerWarps * 32) {
        const int e = idx * 2;
        const int h = e / D;
        float o0 = 0.f, o1 = 0.f;
#pragma unroll
        for (int q = 0; q < kConsumerWarps; ++q) {
          o0 += red[q * G * D + e];
          o1 += red[q * G * D + e + 1];
        }
        const float inv = 1.f / lstat[h];
        *reinterpret_cast<uint32_t *>(p.out + ((int64_t)s * Hq + h0) * D + e) =
            pack_bf16x2(o0 * inv, o1 * inv);
      }
    } else {
      float *po = p.part_o + ((int64_t)gblk * Hq + h0) * D;
      for (int idx = tid; idx < G * D / 4; idx += kConsumerWarps * 32) {
        const int e = idx * 4;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < kConsumerWarps; ++q) {
          const float4 x = *reinterpret_cast<const float4 *>(red + q * G * D + e);
          o.x += x.x;
          o.y += x.y;
          o.z += x.z;
          o.w += x.w;
        }
        *reinterpret_cast<float4 *>(po + e) = o;
      }
      if (tid < G) {
        p.part_ml[((int64_t)gblk * Hq + h0 + tid) * 2] = mstat[tid];
        p.part_ml[((int64_t)gblk * Hq + h0 + tid) * 2 + 1] = lstat[tid];
      }
    }
    // All consumer warps agree on whether to stop (a wait ran out).
    if (named_bar_or(1, kConsumerWarps * 32, *abort_flag != 0)) {
      if (tid == 0) flag_status(p.status, PKV_DEV_TIMEOUT);
      break;
    }
  }
}

// Split-K merge: one CTA per (sequence, kv head) with more than one item (partial).
// M = max_b m_b;  O = sum_b 2^(m_b - M) o_b / sum_b 2^(m_b - M) l_b  (log2 units).
// Threads are split into groups that take interleaved partials; each thread
// merges its partials in one pass (running max, rescaling what it has so
// far), so all of its loads are independent, and the groups are combined in
// shared memory the same way.
constexpr int kMergeThreads = 256;
// For small batches whose merge CTAs all fit beside the split-K grid, a
// merge CTA finds its sequence's partials from context_lens itself (the same
// block counts as the split-K grid) while that grid is still running, rather
// than reading the published prefix after it: measured, the 64-sequence
// decode batch 60.2 -> 59.6 us; the 256-sequence long decode (2048 merge
// CTAs, most of them scheduled only after the split-K grid) 354 -> 362 us.
constexpr int kMergeLocalSeqs = 128;
constexpr int kMergeLocalCtasPerSm = 4;

template <int D, int G, bool kLocal>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const DecodeParams p) {
  constexpr int V4 = G * D / 4;  // float4 outputs per (sequence, kv head)
  constexpr int GR = V4 >= kMergeThreads ? 1 : kMergeThreads / V4;
  __shared__ float4 red[GR][V4];
  __shared__ float sM[GR][G], sL[GR][G];
  const int Hkv = p.num_kv_heads;
  const int Hq = p.num_q_heads;
  const int s = blockIdx.x / Hkv;
  const int j = blockIdx.x - s * Hkv;
  const int tid = threadIdx.x;
  int pb0 = 0, nblk = 0;
  if constexpr (kLocal) {
    // (A local merge always follows the split-K kernel's one-block form, so
    // a sequence's partials are its blocks.)
    __shared__ int sRed[3][kMergeThreads / 32];
    // context_lens is an input of the call: the split-K grid never writes it.
    int before = 0, total = 0, bad = 0;
    for (int i = tid; i < p.num_seqs; i += kMergeThreads) {
      const int nb = seq_blocks(p.context_lens[i], p.block_size, p.max_blocks_per_seq, &bad);
      total += nb;
      if (i < s) before += nb;
      if (i == s) nblk = nb;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      before += __shfl_xor_sync(0xffffffffu, before, o);
      total += __shfl_xor_sync(0xffffffffu, total, o);
      nblk += __shfl_xor_sync(0xffffffffu, nblk, o);
    }
    if ((tid & 31) == 0) {
      sRed[0][tid >> 5] = before;
      sRed[1][tid >> 5] = total;
      sRed[2][tid >> 5] = nblk;
    }
    __syncthreads();
    before = 0;
    total = 0;
    nblk = 0;
#pragma unroll
    for (int w = 0; w < kMergeThreads / 32; ++w) {
      before += sRed[0][w];
      total += sRed[1][w];
      nblk += sRed[2][w];
    }
    // Nothing to merge: one block, or the split-K grid refused the call for
    // want of workspace (it then leaves every partial unwritten).
    if (nblk <= 1 || (int64_t)total > p.max_total_blocks) return;
    pb0 = before;
  }
  // Partials are complete once the split-K grid has finished.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if constexpr (!kLocal) {
    pb0 = p.seq_prefix[s];
    nblk = p.seq_prefix[s + 1] - pb0;
    if (nblk <= 1) return;  // single-item sequences were finished by the split-K grid
  }
  if (pb0 < 0 || (int64_t)pb0 + nblk > p.max_total_blocks) return;  // never index past the workspace
  const int h0 = j * G;
  const int v = tid % V4;
  const int g = tid / V4;
  const int e = v * 4;
  const int h = e / D;
  float M = -INFINITY, L = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  if (g < GR) {
#pragma unroll 4
    for (int b = g; b < nblk; b += GR) {
      const int64_t row = (int64_t)(pb0 + b) * Hq + h0 + h;
      const float2 ml = __ldcg(reinterpret_cast<const float2 *>(p.part_ml + row * 2));
      const float4 x = __ldcg(reinterpret_cast<const float4 *>(p.part_o + row * D + (e - h * D)));
      const float Mn = fmaxf(M, ml.x);
      const float a = fast_exp2(M - Mn);  // 0 while nothing is merged yet (M = -inf)
      const float w = fast_exp2(ml.x - Mn);
      o.x = fmaf(w, x.x, o.x * a);
      o.y = fmaf(w, x.y, o.y * a);
      o.z = fmaf(w, x.z, o.z * a);
      o.w = fmaf(w, x.w, o.w * a);
      L = fmaf(w, ml.y, L * a);
      M = Mn;
    }
    red[g][v] = o;
    if (e - h * D == 0) {
      sM[g][h] = M;
      sL[g][h] = L;
    }
  }
  __syncthreads();
  if (tid >= V4) return;
  // Combine the groups (a group without partials has M = -inf: factor 0).
  float Mf = -INFINITY;
#pragma unroll
  for (int q = 0; q < GR; ++q) Mf = fmaxf(Mf, sM[q][h]);
  float Lf = 0.f;
  o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int q = 0; q < GR; ++q) {
    const float c = fast_exp2(sM[q][h] - Mf);
    const float4 x = red[q][v];
    o.x = fmaf(c, x.x, o.x);
    o.y = fmaf(c, x.y, o.y);
    o.z = fmaf(c, x.z, o.z);
    o.w = fmaf(c, x.w, o.w);
    Lf = fmaf(c, sL[q][h], Lf);
  }
  const float inv = 1.f / Lf;
  uint2 packed;
  packed.x = pack_bf16x2(o.x * inv, o.y * inv);
  packed.y = pack_bf16x2(o.z * inv, o.w * inv);
  *reinterpret_cast<uint2 *>(p.out + ((int64_t)s * Hq + h0) * D + e) = packed;
}

template <int D, int G>
pkv_status launch_decode(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &prm,
                         int64_t max_items, cudaStream_t stream) {
  const DecodeSmem lay(D, G, prm.block_size, prm.num_seqs);
  const int smem = lay.total + 1024;  // + alignment slack
  int ctas_per_sm = 0;
  const int64_t merge_grid = (int64_t)prm.num_seqs * prm.num_kv_heads;
  const int sms = device_sm_count();
  if (sms <= 0) return PKV_ERR_CUDA;
  const bool local =
      prm.num_seqs <= kMergeLocalSeqs && merge_grid <= (int64_t)kMergeLocalCtasPerSm * sms;
  // Items may span two blocks only when the merge reads the published prefix
  // and there can be enough items for it (then the kernel decides).
  const bool span = !local && max_items >= (int64_t)kSpanRounds * 3 * sms;
  const void *kfn = span ? (const void *)paged_decode_kernel<D, G, true>
                         : (const void *)paged_decode_kernel<D, G, false>;
  if (!kernel_smem_setup(kfn, kThreads, smem, &ctas_per_sm)) return PKV_ERR_CUDA;
  int64_t grid = (int64_t)sms * ctas_per_sm;
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  if (span)
    paged_decode_kernel<D, G, true><<<(unsigned)grid, kThreads, smem, stream>>>(tk, tv, prm);
  else
    paged_decode_kernel<D, G, false><<<(unsigned)grid, kThreads, smem, stream>>>(tk, tv, prm);
  if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  if (prm.max_blocks_per_seq <= 1) return PKV_OK;  // nothing can need a merge
  // The merge grid is launched as a programmatic dependent of the split-K
  // grid: it may be scheduled early and waits (griddepcontrol.wait) for the
  // split-K grid's completion before reading the partials.
  if (merge_grid > 0x7FFFFFFFLL) return PKV_ERR_INVALID_ARG;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)merge_grid);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = local ? cudaLaunchKernelEx(&cfg, decode_merge_kernel<D, G, true>, prm)
                              : cudaLaunchKernelEx(&cfg, decode_merge_kernel<D, G, false>, prm);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  return launch_status();
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace
}  // namespace pkv

extern "C" size_t pkv_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                            int head_dim, int64_t max_total_blocks) {
  using pkv::align256;
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_total_blocks < 0)
    return 0;
  // Sizes whose product would not fit a size_t (the factors are bounded first
  // so that the per-block product itself cannot wrap) have no workspace.
  if (num_q_heads > (1 << 16) || head_dim > (1 << 16)) return 0;
  const size_t per_block = (size_t)num_q_heads * ((size_t)head_dim + 2) * 4;
  if ((uint64_t)max_total_blocks > (SIZE_MAX / 2 - (size_t)num_seqs * 4 - 1024) / per_block)
    return 0;
  return 256 /* item counter */ + align256((size_t)(num_seqs + 1) * 4) +
         align256((size_t)max_total_blocks * num_q_heads * 2 * 4) +
         align256((size_t)max_total_blocks * num_q_heads * head_dim * 4);
}

namespace pkv {
namespace {

// Shared by the plain and the fused-store decode entry points (the fused one
// passes the new tokens' rows, their slots and writable cache pointers).
pkv_status decode_call(uint16_t *out, const uint16_t *q, const uint16_t *k_cache,
                       const uint16_t *v_cache, const int32_t *block_tables,
                       const int32_t *context_lens, int num_seqs, int num_q_heads,
                       int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                       int64_t num_blocks, int64_t max_total_blocks, float scale, void *workspace,
                       size_t workspace_bytes, int32_t *dev_status, void *stream,
                       const uint16_t *new_k, const uint16_t *new_v, const int32_t *new_slots,
                       uint16_t *k_cache_w, uint16_t *v_cache_w) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      block_size <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || max_total_blocks < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  const int G = num_q_heads / num_kv_heads;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_ERR_UNSUPPORTED;
  if (block_size != 64 && block_size != 128 && block_size != 256 && block_size != 512)
    return PKV_ERR_UNSUPPORTED;
  if (num_seqs > kMaxSeqs) return PKV_ERR_UNSUPPORTED;
  if (!isfinite(scale)) return PKV_ERR_INVALID_ARG;  // NaN or infinite
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  // The kernel keeps per-sequence block offsets and lengths in shared memory:
  // batches whose layout would not fit are refused before any launch.
  if (DecodeSmem(head_dim, G, block_size, num_seqs).total + 1024 > kMaxDynamicSmem)
    return PKV_ERR_UNSUPPORTED;
  const size_t need =
      pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_total_blocks);
  if (need == 0) return PKV_ERR_INVALID_ARG;  // a workspace that size cannot be addressed
  if (workspace == nullptr || workspace_bytes < need ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return PKV_ERR_WORKSPACE;

  DecodeParams prm;
  prm.out = out;
  prm.q = q;
  prm.block_tables = block_tables;
  prm.context_lens = context_lens;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  prm.ctl = reinterpret_cast<unsigned int *>(ws);
  ws += 256;
  prm.seq_prefix = reinterpret_cast<int32_t *>(ws);
  ws += align256((size_t)(num_seqs + 1) * 4);
  prm.part_ml = reinterpret_cast<float *>(ws);
  ws += align256((size_t)max_total_blocks * num_q_heads * 2 * 4);
  prm.part_o = reinterpret_cast<float *>(ws);
  prm.status = dev_status;
  prm.num_blocks = num_blocks;
  prm.max_total_blocks = max_total_blocks;
  prm.num_seqs = num_seqs;
  prm.num_q_heads = num_q_heads;
  prm.num_kv_heads = num_kv_heads;
  prm.block_size = block_size;
  prm.max_blocks_per_seq = max_blocks_per_seq;
  prm.qscale = scale * kLog2e;
  prm.span_ok = 1;
  prm.new_k = new_k;
  prm.new_v = new_v;
  prm.new_slots = new_slots;
  prm.k_cache_w = k_cache_w;
  prm.v_cache_w = v_cache_w;
  prm.k_cache_r = k_cache;
  prm.v_cache_r = v_cache;

  // K/V cache as a 4-D tensor {D, Hkv, block_size, num_blocks}; a box is one
  // kv head's 64 consecutive tokens of one block.
  const uint64_t dims[4] = {(uint64_t)head_dim, (uint64_t)num_kv_heads, (uint64_t)block_size,
                            (uint64_t)num_blocks};
  const uint64_t strides[3] = {(uint64_t)head_dim * 2, (uint64_t)num_kv_heads * head_dim * 2,
                               (uint64_t)block_size * num_kv_heads * head_dim * 2};
  const uint32_t box[4] = {(uint32_t)head_dim, 1u, (uint32_t)kTile, 1u};
  CUtensorMap tk, tv;
  if (!encode_bf16_map(&tk, k_cache, 4, dims, strides, box, false) ||
      !encode_bf16_map(&tv, v_cache, 4, dims, strides, box, false))
    return PKV_ERR_CUDA;

  int64_t max_items = (int64_t)num_seqs * max_blocks_per_seq;
  if (max_items > max_total_blocks) max_items = max_total_blocks;
  max_items *= num_kv_heads;
  if (max_items < 1) max_items = 1;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
#define PKV_DECODE_CASE(DD, GG) \
  if (head_dim == DD && G == GG) return launch_decode<DD, GG>(tk, tv, prm, max_items, st);
  PKV_DECODE_CASE(64, 1)
  PKV_DECODE_CASE(64, 2)
  PKV_DECODE_CASE(64, 4)
  PKV_DECODE_CASE(64, 8)
  PKV_DECODE_CASE(128, 1)
  PKV_DECODE_CASE(128, 2)
  PKV_DECODE_CASE(128, 4)
  PKV_DECODE_CASE(128, 8)
#undef PKV_DECODE_CASE
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_paged_decode_attn(uint16_t *out, const uint16_t *q,
                                            const uint16_t *k_cache, const uint16_t *v_cache,
                                            const int32_t *block_tables,
                                            const int32_t *context_lens, int num_seqs,
                                            int num_q_heads, int num_kv_heads, int head_dim,
                                            int block_size, int max_blocks_per_seq,
                                            int64_t num_blocks, int64_t max_total_blocks,
                                            float scale, void *workspace, size_t workspace_bytes,
                                            int32_t *dev_status, void *stream) {
  return pkv::decode_call(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                          num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                          num_blocks, max_total_blocks, scale, workspace, workspace_bytes,
                          dev_status, stream, nullptr, nullptr, nullptr, nullptr, nullptr);
}

extern "C" pkv_status pkv_paged_decode_store_attn(
    uint16_t *out, const uint16_t *q, const uint16_t *new_k, const uint16_t *new_v,
    const int32_t *slot_mapping, uint16_t *k_cache, uint16_t *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq, int64_t num_blocks,
    int64_t max_total_blocks, float scale, void *workspace, size_t workspace_bytes,
    int32_t *dev_status, void *stream) {
  using namespace pkv;
  if (num_seqs > 0 && (!new_k || !new_v || !slot_mapping || !aligned16(new_k) || !aligned16(new_v)))
    return PKV_ERR_INVALID_ARG;
  return decode_call(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                     num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
                     max_total_blocks, scale, workspace, workspace_bytes, dev_status, stream,
                     new_k, new_v, slot_mapping, k_cache, v_cache);
}

// ---------------------------------------------------------------------------
// Allocation-free variant.
//
// Some callers cannot hand this library a device workspace: a host framework
// whose allocator owns all device memory and offers no hook, a plugin that is
// not allowed to allocate inside the host process, or a serving loop that
// must not call cudaMalloc/cudaFree on its latency path because those calls
// synchronise the device.  For them, the decode scratch (sequence prefix and split-K
// partials) lives in one fixed array in the library's own device memory.
// ---------------------------------------------------------------------------

namespace pkv {
namespace {
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;  // 16 MiB per device
}  // namespace
}  // namespace pkv

// Loaded with the library on every GPU it runs on and held until exit.
static __device__ __align__(256) uint8_t pkv_decode_scratch[pkv::kNoAllocScratchBytes];

namespace pkv {
namespace {

std::mutex g_scratch_mu;
void *g_scratch_ptr[64] = {nullptr};

// Device address of pkv_decode_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
pkv_status scratch_for_current_device(void **ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= 64) return PKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, pkv_decode_scratch) != cudaSuccess || p == nullptr)
      return PKV_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_paged_decode_attn_noalloc(
    uint16_t *out, const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq, int64_t num_blocks,
    int64_t max_total_blocks, float scale, int32_t *dev_status, void *stream) {
  using namespace pkv;
  if (max_total_blocks > (int64_t)kNoAllocScratchBytes) return PKV_ERR_WORKSPACE;
  const size_t need =
      pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_total_blocks);
  if (need == 0) {
    // Bad sizes or an empty batch: the regular entry point reports it.
    return pkv_paged_decode_attn(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                 num_q_heads, num_kv_heads, head_dim, block_size,
                                 max_blocks_per_seq, num_blocks, max_total_blocks, scale,
                                 nullptr, 0, dev_status, stream);
  }
  if (need > kNoAllocScratchBytes) return PKV_ERR_WORKSPACE;
  void *scratch = nullptr;
  const pkv_status st = scratch_for_current_device(&scratch);
  if (st != PKV_OK) return st;
  // The array keeps the previous call's contents.  Its work counter (first
  // 256 bytes) starts at zero when the library loads and every call leaves
  // it at zero; the rest is written by each call before it is read.
  return pkv_paged_decode_attn(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                               num_q_heads, num_kv_heads, head_dim, block_size,
                               max_blocks_per_seq, num_blocks, max_total_blocks, scale, scratch,
                               kNoAllocScratchBytes, dev_status, stream);
}

// ---------------------------------------------------------------------------
// Test-only fault injection for the bounded waits of the decode kernel.
// ---------------------------------------------------------------------------

extern "C" pkv_status pkv_test_decode_fault(int64_t wait_limit_ns, int withhold_tile) {
  if (wait_limit_ns <= 0 || withhold_tile < -1) return PKV_ERR_INVALID_ARG;
  const unsigned long long limit = (unsigned long long)wait_limit_ns;
  if (cudaMemcpyToSymbol(pkv::g_wait_limit_ns, &limit, sizeof(limit)) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (cudaMemcpyToSymbol(pkv::g_decode_withhold_tile, &withhold_tile, sizeof(int)) != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}
