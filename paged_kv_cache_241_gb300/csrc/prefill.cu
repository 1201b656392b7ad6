// prefill.cu -- causal varlen prefill attention over the paged cache (tcgen05).
//
// Prefill processes whole prompts at once and is compute-dense, unlike decode
// (CSDN essay "from nanoVLLM to vLLM", Mountain 3 and the study route's note
// on the attention/ module).  Its keys and values, including a prefix that was
// cached earlier, live in fixed 256-token blocks reached through the block
// table (same essay, Mountain 1; nano-vllm hub page, "core tech 4").  The
// result is standard softmax attention; like FlashAttention the kernel only
// reorders the computation into on-chip tiles (same essay, Mountain 3).
//
// Design (GB300):
//  * One CTA per (sequence, 128-query tile, pair of query heads of one GQA
//    group); CTAs are ordered sequence-major (heaviest tiles of a sequence
//    first) so that concurrent CTAs reuse a sequence's K/V from L2.  The two
//    heads share every K/V tile.
//  * Warp 0 issues TMA: the Q tiles once, then K and V tiles of 64 keys as
//    128B-swizzled 4-D boxes {64 dims, 1 head, 64 tokens, 1 block}, the block
//    id coming from the block table, into a 4-stage ring.
//  * Warp 1 issues tcgen05.mma: S_h = Q_h K^T (M=128, N=64) into tensor memory,
//    then O_h += P_h V (M=128, N=D) with V as an MN-major operand.
//  * Warps 2-5 (one thread per query row) read S from tensor memory, apply the
//    causal mask offset by the cached length, run the online softmax in fp32
//    (log2 domain), rescale O in tensor memory when the row max grows, write
//    P as bf16 into shared memory in the MMA's swizzled layout, and finally
//    normalise O and store bf16 rows.
#include <math.h>

#include "host_common.h"
#include "pkv_common.cuh"

namespace pkv {
namespace {

constexpr int BM = 128;  // query rows per tile (MMA M)
constexpr int BN = 64;   // keys per tile
// Warp 0: Q/K TMA producer; warp 1: S = QK^T MMA issuer; then one 4-warp
// softmax group per head; then the V TMA producer and the P.V MMA issuer.
template <int NH>
constexpr int threads_for() { return 128 + 128 * NH; }
constexpr float kLog2e = 1.4426950408889634f;

struct PrefillParams {
  uint16_t *out;
  const int32_t *block_tables;
  const int32_t *cu_q;
  const int32_t *cu_k;
  int32_t *status;
  int64_t num_blocks;
  int64_t total_q;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int block_size;
  int max_blocks_per_seq;
  int q_tiles;  // ceil(max_seqlen_q / BM)
  float qscale; // scale * log2(e)
};

template <int D, int NH>
struct PrefillLayout {
  static constexpr int kQBytes = BM * D * 2;   // one head's Q tile
  static constexpr int kKVBytes = BN * D * 2;  // one K or V tile
  // Ring depths: the K/V slots that fit next to Q in 227 KiB of shared
  // memory (at most 12).  A K slot is held until its S MMAs finish, a V slot
  // until its P.V has run, so V gets the larger share.
  static constexpr int kSlots0 = (232448 - 2048 - NH * kQBytes) / kKVBytes;
  static constexpr int kSlots = kSlots0 < 12 ? kSlots0 : 12;
  static constexpr int kKStages = kSlots * 2 / 5;
  static constexpr int kVStages = kSlots - kKStages;
  static constexpr int q = 0;
  static constexpr int k = q + NH * kQBytes;
  static constexpr int v = k + kKStages * kKVBytes;
  static constexpr int bars = v + kVStages * kKVBytes;
  // barriers: q_full, k_full[SK], v_full[SV], k_empty[SK], v_empty[SV],
  // s_full[NH][2], s_free[NH][2], p_full[NH], o_done[NH], drain
  static_assert(kKStages >= 2 && kVStages >= 2, "rings too shallow");
  static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 4 * NH + 2 * NH + 1;
  static constexpr int misc = bars + kNumBars * 8;  // tmem address, abort flag
  static constexpr int total = misc + 16;
  static constexpr int kCols = NH * D + 2 * NH * BN;  // O per head + two S buffers per head
  static constexpr int kTmemCols = kCols <= 128 ? 128 : (kCols <= 256 ? 256 : 512);
};

// Tensor-memory columns (fp32, lane = query row): O_h at kO + h*D; the two S
// buffers of head h at kS + (2h + b)*BN, b = tile index & 1.  The softmax
// overwrites S(jt) in place with P(jt) as bf16 pairs (its first BN/2
// columns), the A operand of that tile's P.V.
template <int D, int NH>
struct TmemCols {
  static constexpr uint32_t kO = 0;
  static constexpr uint32_t kS = NH * D;
};

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
  const bool ok = mbar_wait_bounded(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

template <int D, int NH>
__global__ void __launch_bounds__(threads_for<NH>(), 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using L = PrefillLayout<D, NH>;
  constexpr int XR = D / 64;  // 128-byte swizzle regions across D
  constexpr int kKStages = L::kKStages;
  constexpr int kVStages = L::kVStages;
  constexpr uint32_t kOCol = TmemCols<D, NH>::kO;
  constexpr uint32_t kSCol = TmemCols<D, NH>::kS;
  constexpr int kVWarp = 2 + 4 * NH;   // V producer warp (after the softmax warpgroups)
  constexpr int kPVWarp = 3 + 4 * NH;  // P.V MMA issuer

  // ---- which tile -------------------------------------------------------
  // Sequence-major order, each sequence's heaviest q tiles first, head groups
  // innermost: CTAs running together share a sequence's K/V in L2.
  const int HG = p.num_q_heads / NH;
  int idx = blockIdx.x;
  const int hg = idx % HG;
  idx /= HG;
  const int tr = idx % p.q_tiles;  // 0 = the sequence's last (heaviest) q tile
  const int s = idx / p.q_tiles;
  const int q_begin = p.cu_q[s];
  const int n = p.cu_q[s + 1] - q_begin;
  const int len_k = p.cu_k[s + 1] - p.cu_k[s];
  const int c = len_k - n;
  if (n <= 0) return;
  const int ntq = (n + BM - 1) / BM;
  if (c < 0 || len_k > p.max_blocks_per_seq * p.block_size || ntq > p.q_tiles ||
      (int64_t)q_begin + n > p.total_q) {
    if (tr == 0 && hg == 0 && threadIdx.x == 0) flag_status(p.status, PKV_DEV_BAD_SEQLEN);
    if (c < 0 || len_k > p.max_blocks_per_seq * p.block_size || (int64_t)q_begin + n > p.total_q)
      return;
  }
  const int t = ntq - 1 - tr;
  if (t < 0) return;
  const int q0 = t * BM;
  const int rows_valid = min(BM, n - q0);
  const int kv_end = min(len_k, c + q0 + rows_valid);  // keys needed by this tile
  const int n_kv = (kv_end + BN - 1) / BN;
  const int h_first = hg * NH;
  const int G = p.num_q_heads / p.num_kv_heads;
  const int kvh = h_first / G;

  // ---- shared memory ----------------------------------------------------
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem + L::q;
  uint8_t *sK = smem + L::k;
  uint8_t *sV = smem + L::v;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bars);
  uint64_t *q_full = bars;
  uint64_t *k_full = bars + 1;
  uint64_t *v_full = k_full + kKStages;
  uint64_t *k_empty = v_full + kVStages;
  uint64_t *v_empty = k_empty + kKStages;
  uint64_t *s_full = v_empty + kVStages;  // [NH][2]
  uint64_t *s_free = s_full + 2 * NH;     // [NH][2]: P.V has read P out of that buffer
  uint64_t *p_full = s_free + 2 * NH;
  uint64_t *o_done = p_full + NH;
  uint64_t *drain = o_done + NH;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::misc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int h = 0; h < NH; ++h) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(&s_full[2 * h + b], 1);
        mbar_init(&s_free[2 * h + b], 1);
      }
      mbar_init(&p_full[h], 128);  // one softmax warpgroup per head
      mbar_init(&o_done[h], 1);
    }
    mbar_init(drain, 2);  // one commit from each MMA issuer
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // Physical block and in-block offset of KV tile jt (bounds-checked).
  auto block_of = [&](int jt, int &off) {
    const int key0 = jt * BN;
    const int lb = key0 / p.block_size;
    off = key0 - lb * p.block_size;
    int blk = p.block_tables[(int64_t)s * p.max_blocks_per_seq + lb];
    if (blk < 0 || (int64_t)blk >= p.num_blocks) {
      flag_status(p.status, PKV_DEV_BAD_BLOCK);
      blk = 0;
    }
    return blk;
  };

  if (warp == 0 || warp == kVWarp) {
    // ============ TMA producers: warp 0 loads Q and K, the last warp V ============
    // The K and V rings turn over independently: a K slot is free once the
    // S MMAs that read it are done, a V slot once its P.V MMAs are done.
    if (lane == 0) {
      const bool is_k = (warp == 0);
      uint64_t *full = is_k ? k_full : v_full;
      uint64_t *empty = is_k ? k_empty : v_empty;
      uint8_t *ring = is_k ? sK : sV;
      const CUtensorMap *map = is_k ? &tm_k : &tm_v;
      const int nst = is_k ? kKStages : kVStages;
      if (is_k) {
        tma_prefetch_map(&tm_q);
        tma_prefetch_map(&tm_k);
        mbar_arrive_expect_tx(q_full, NH * L::kQBytes);
        for (int h = 0; h < NH; ++h)
          for (int x = 0; x < XR; ++x)
            tma_load_3d(sQ + h * L::kQBytes + x * BM * 128, &tm_q, q_full, x * 64, h_first + h,
                        q_begin + q0);
      } else {
        tma_prefetch_map(&tm_v);
      }
      int issued = 0;
      for (int jt = 0; jt < n_kv; ++jt) {
        const int st = jt % nst;
        if (jt >= nst && !mbar_wait_bounded(&empty[st], ((jt / nst) - 1) & 1, abort_flag))
          break;
        int off;
        const int blk = block_of(jt, off);
        mbar_arrive_expect_tx(&full[st], L::kKVBytes);
        for (int x = 0; x < XR; ++x)
          tma_load_4d(ring + st * L::kKVBytes + x * BN * 128, map, &full[st], x * 64, kvh, off,
                      blk);
        issued = jt + 1;
      }
      // Do not leave while copies into this CTA's shared memory are in flight.
      if (is_k && !mbar_wait_bounded(q_full, 0, nullptr)) flag_status(p.status, PKV_DEV_TIMEOUT);
      for (int i = max(0, issued - nst); i < issued; ++i)
        if (!mbar_wait_bounded(&full[i % nst], (i / nst) & 1, nullptr))
          flag_status(p.status, PKV_DEV_TIMEOUT);
    }
  } else if (warp == 1 || warp == kPVWarp) {
    // ============ MMA issuers: warp 1 issues S = QK^T, the last warp O += PV ============
    // Two issuing threads keep the tensor pipe fed while either one waits on
    // a barrier (its queue of issued MMAs is short).  Shared-memory matrix
    // descriptors are built once; an MMA only adds the operand's offset to
    // the address field (bits 0-13, bytes / 16).
    if (lane == 0) {
      bool ok = true;
      if (warp == 1) {
        constexpr uint32_t idesc_s = umma_idesc_bf16(BM, BN, false, false);
        const uint64_t dq = umma_desc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dk = umma_desc_sw128(smem_u32(sK), 16, 1024);
        ok = mbar_wait_bounded(q_full, 0, abort_flag);
        // Per tile jt: S_h(jt) for every head into S buffer jt & 1 once K(jt)
        // is in and P.V(jt - 2) has read P_h(jt - 2) out of that buffer.
        for (int jt = 0; jt < n_kv && ok; ++jt) {
          const int st = jt % kKStages;
          ok = mbar_wait_bounded(&k_full[st], (jt / kKStages) & 1, abort_flag);
          const uint64_t dk_st = dk + (uint64_t)((st * L::kKVBytes) >> 4);
#pragma unroll
          for (int h = 0; h < NH && ok; ++h) {
            uint64_t *sf = &s_free[2 * h + (jt & 1)];
            if (jt >= 2) ok = mbar_wait_bounded(sf, ((jt - 2) >> 1) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t d = tmem + kSCol + (2 * h + (jt & 1)) * BN;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk & 3) * 32;
              umma_bf16(d, dq + (uint64_t)((h * L::kQBytes + (kk / 4) * BM * 128 + off) >> 4),
                        dk_st + (uint64_t)(((kk / 4) * BN * 128 + off) >> 4), idesc_s,
                        kk > 0 ? 1u : 0u);
            }
            umma_commit(&s_full[2 * h + (jt & 1)]);
          }
          if (ok) umma_commit(&k_empty[st]);
        }
      } else {
        constexpr uint32_t idesc_o = umma_idesc_bf16(BM, D, false, true);
        const uint64_t dv = umma_desc_sw128(smem_u32(sV), BN * 128, 1024);
        // Per tile jt, in head order: O_h += P_h(jt) V(jt) (P from tensor
        // memory) once V(jt) is in and the head's P is written; then the S
        // buffer and the V slot are released.  Head order also keeps every
        // head's last P.V behind warpgroup 0, which clears the V rows past
        // the context before it publishes its P.
        for (int jt = 0; jt < n_kv && ok; ++jt) {
          const int pst = jt % kVStages;
          ok = mbar_wait_bounded(&v_full[pst], (jt / kVStages) & 1, abort_flag);
          const uint64_t dv_st = dv + (uint64_t)((pst * L::kKVBytes) >> 4);
#pragma unroll
          for (int h = 0; h < NH && ok; ++h) {
            ok = mbar_wait_bounded(&p_full[h], jt & 1, abort_flag);
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t pa = tmem + kSCol + (2 * h + (jt & 1)) * BN;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              umma_bf16_tmem_a(tmem + kOCol + h * D, pa + kk * 8,
                               dv_st + (uint64_t)((kk * 16 * 128) >> 4), idesc_o,
                               (jt > 0 || kk > 0) ? 1u : 0u);
            umma_commit(&o_done[h]);
            umma_commit(&s_free[2 * h + (jt & 1)]);
          }
          if (ok) umma_commit(&v_empty[pst]);
        }
      }
      // Wait for the MMAs of both issuers before tensor memory is freed.
      umma_commit(drain);
      if (!mbar_wait_bounded(drain, 0, nullptr)) flag_status(p.status, PKV_DEV_TIMEOUT);
    }
  } else {
    // ================= softmax / epilogue: one warpgroup per head =================
    const int h = (warp - 2) >> 2;  // the head this warpgroup serves
    const int quarter = warp & 3;   // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int key_limit = min(c + q0 + row, len_k - 1);  // last key this row may see
    const float qs = p.qscale;
    // Running max in log2 units.  It is only raised (and O rescaled) when a
    // tile's max exceeds it by more than 8, so P stays <= 2^8; l and O share
    // the same reference, so the final O / l is unchanged.
    float m_ref = -INFINITY;
    float l_run = 0.f;
    bool ok = true;
    for (int jt = 0; jt < n_kv && ok; ++jt) {
      const int key0 = jt * BN;
      ok = warp_wait(&s_full[2 * h + (jt & 1)], (jt >> 1) & 1, abort_flag);
      if (!ok) break;
      tc_fence_after_sync();
      float sv[BN];
      static_assert(BN == 64, "S is read with one 64-column TMEM load");
      const uint32_t s_addr = tmem + lane_base + kSCol + (2 * h + (jt & 1)) * BN;
      tmem_load64(s_addr, sv);
      // Tile max of the scaled logits over this row's visible keys (4-way tree).
      const bool full_row = key0 + BN - 1 <= key_limit;
      float mt;
      {
        float e0 = -INFINITY, e1 = -INFINITY, e2 = -INFINITY, e3 = -INFINITY;
        if (qs >= 0.f) {
          if (full_row) {
#pragma unroll
            for (int i = 0; i < BN; i += 4) {
              e0 = fmaxf(e0, sv[i]);
              e1 = fmaxf(e1, sv[i + 1]);
              e2 = fmaxf(e2, sv[i + 2]);
              e3 = fmaxf(e3, sv[i + 3]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < BN; ++i)
              if (key0 + i <= key_limit) e0 = fmaxf(e0, sv[i]);
          }
          mt = fmaxf(fmaxf(e0, e1), fmaxf(e2, e3)) * qs;
        } else {
          e0 = INFINITY;
#pragma unroll
          for (int i = 0; i < BN; ++i)
            if (key0 + i <= key_limit) e0 = fminf(e0, sv[i]);
          mt = e0 * qs;
        }
      }
      // Key 0 is in the first tile and visible to every row, so the first tile
      // sets a finite max (the -inf guard keeps a row with no visible key at
      // alpha = 0 instead of NaN).
      float alpha = 1.f;
      if (jt == 0 || mt > m_ref + 8.f) {
        const float m_new = fmaxf(m_ref, mt);
        alpha = (m_ref == -INFINITY) ? 0.f : fast_exp2(m_ref - m_new);
        m_ref = m_new;
      }
      float rs;
      {
        float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
        if (full_row) {
#pragma unroll
          for (int i = 0; i < BN; i += 4) {
            sv[i] = fast_exp2(fmaf(sv[i], qs, -m_ref));
            sv[i + 1] = fast_exp2(fmaf(sv[i + 1], qs, -m_ref));
            sv[i + 2] = fast_exp2(fmaf(sv[i + 2], qs, -m_ref));
            sv[i + 3] = fast_exp2(fmaf(sv[i + 3], qs, -m_ref));
            r0 += sv[i];
            r1 += sv[i + 1];
            r2 += sv[i + 2];
            r3 += sv[i + 3];
          }
        } else {
#pragma unroll
          for (int i = 0; i < BN; i += 4) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              sv[i + u] =
                  (key0 + i + u <= key_limit) ? fast_exp2(fmaf(sv[i + u], qs, -m_ref)) : 0.f;
            r0 += sv[i];
            r1 += sv[i + 1];
            r2 += sv[i + 2];
            r3 += sv[i + 3];
          }
        }
        rs = (r0 + r1) + (r2 + r3);
      }
      if (jt > 0 && __any_sync(0xffffffffu, alpha < 1.f)) {
        // O is rescaled once P.V(jt - 1) has landed in it (P.V(jt) waits for
        // this tile's P).  P.V(jt - 2) is complete (S(jt) waited for it), so
        // the parity wait cannot alias.
        ok = warp_wait(&o_done[h], (jt - 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after_sync();
        {
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            float ov[32];
            const uint32_t oa = tmem + lane_base + kOCol + h * D + cc * 32;
            tmem_load32(oa, ov);
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] *= alpha;
            tmem_store32(oa, ov);
          }
        }
      }
      l_run = l_run * alpha + rs;
      if (h == 0 && key0 + BN > len_k) {
        // Keys past the context may hold stale bits (even NaN); P is zero
        // there, but 0 * NaN is not, so clear those V rows first.  (The MMA
        // thread issues every head's last P.V after this warpgroup's arrival.)
        ok = warp_wait(&v_full[jt % kVStages], (jt / kVStages) & 1, abort_flag);
        if (!ok) break;
        const int first = len_k - key0;
        uint8_t *vt = sV + (jt % kVStages) * L::kKVBytes;
        const int nchunks = (BN - first) * 8 * XR;  // 16-byte chunks to clear
        for (int i = row; i < nchunks; i += 128) {
          const int x = i / ((BN - first) * 8);
          const int rem = i - x * (BN - first) * 8;
          const int rr = first + rem / 8;
          *reinterpret_cast<uint4 *>(vt + x * BN * 128 + rr * 128 + (rem & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();  // the MMA reads these rows through the async proxy
      }
      // P (bf16 pairs) over the first BN/2 columns of this tile's S buffer.
      {
        float pw[BN / 2];
#pragma unroll
        for (int i = 0; i < BN / 2; ++i) pw[i] = __uint_as_float(pack_bf16x2(sv[2 * i], sv[2 * i + 1]));
        static_assert(BN / 2 == 32, "P is written with one 32-column TMEM store");
        tmem_store32(s_addr, pw);
      }
      tc_fence_before_sync();
      mbar_arrive(&p_full[h]);
    }
    // Epilogue: O / l -> bf16 rows, once the last P.V is in O.  P.V(n_kv - 3)
    // is complete, so waiting on n_kv - 2 then n_kv - 1 cannot alias.
    if (ok && n_kv >= 2) ok = warp_wait(&o_done[h], (n_kv - 2) & 1, abort_flag);
    if (ok) ok = warp_wait(&o_done[h], (n_kv - 1) & 1, abort_flag);
    if (ok) {
      tc_fence_after_sync();
      const float inv = 1.f / l_run;
      uint16_t *dst = p.out + ((int64_t)(q_begin + q0 + row) * p.num_q_heads + h_first + h) * D;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        float ov[32];
        tmem_load32(tmem + lane_base + kOCol + h * D + cc * 32, ov);
        if (row < rows_valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 w;
            w.x = pack_bf16x2(ov[i] * inv, ov[i + 1] * inv);
            w.y = pack_bf16x2(ov[i + 2] * inv, ov[i + 3] * inv);
            w.z = pack_bf16x2(ov[i + 4] * inv, ov[i + 5] * inv);
            w.w = pack_bf16x2(ov[i + 6] * inv, ov[i + 7] * inv);
            *reinterpret_cast<uint4 *>(dst + cc * 32 + i) = w;
          }
        }
      }
    }
    tc_fence_before_sync();
  }

  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) flag_status(p.status, PKV_DEV_TIMEOUT);
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int D, int NH>
pkv_status launch_prefill(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                          const PrefillParams &prm, cudaStream_t stream) {
  using L = PrefillLayout<D, NH>;
  static int smem = 0;
  if (smem == 0) {
    int bytes = L::total + 1024;
    // Resident CTAs per SM must not ask for more than 512 TMEM columns in
    // total, or tcgen05.alloc would stall: pad shared memory to cap occupancy.
    const int max_ctas = 512 / L::kTmemCols;
    const int per_sm = 228 * 1024;
    const int min_bytes = per_sm / (max_ctas + 1) + 1;
    if (bytes < min_bytes) bytes = min_bytes;
    if (cudaFuncSetAttribute(paged_prefill_kernel<D, NH>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
      return PKV_ERR_CUDA;
    smem = bytes;
  }
  const int64_t grid = (int64_t)prm.q_tiles * prm.num_seqs * (prm.num_q_heads / NH);
  if (grid > 0x7FFFFFFFLL) return PKV_ERR_INVALID_ARG;
  paged_prefill_kernel<D, NH><<<(unsigned)grid, threads_for<NH>(), smem, stream>>>(tq, tk, tv, prm);
  return launch_status();
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_paged_prefill_attn(uint16_t *out, const uint16_t *q,
                                             const uint16_t *k_cache, const uint16_t *v_cache,
                                             const int32_t *block_tables,
                                             const int32_t *cu_seqlens_q,
                                             const int32_t *cu_seqlens_k, int num_seqs,
                                             int64_t total_q, int max_seqlen_q, int num_q_heads,
                                             int num_kv_heads, int head_dim, int block_size,
                                             int max_blocks_per_seq, int64_t num_blocks,
                                             float scale, int32_t *dev_status, void *stream) {
  using namespace pkv;
  if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0 || num_q_heads <= 0 ||
      num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || max_blocks_per_seq <= 0 ||
      num_blocks <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  const int G = num_q_heads / num_kv_heads;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_ERR_UNSUPPORTED;
  if (block_size != 64 && block_size != 128 && block_size != 256 && block_size != 512)
    return PKV_ERR_UNSUPPORTED;
  if (!(scale == scale)) return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0) return PKV_OK;
  if (total_q > 0x7FFFFFFFLL) return PKV_ERR_UNSUPPORTED;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !cu_seqlens_q || !cu_seqlens_k)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;

  PrefillParams prm;
  prm.out = out;
  prm.block_tables = block_tables;
  prm.cu_q = cu_seqlens_q;
  prm.cu_k = cu_seqlens_k;
  prm.status = dev_status;
  prm.num_blocks = num_blocks;
  prm.total_q = total_q;
  prm.num_seqs = num_seqs;
  prm.num_q_heads = num_q_heads;
  prm.num_kv_heads = num_kv_heads;
  prm.block_size = block_size;
  prm.max_blocks_per_seq = max_blocks_per_seq;
  prm.q_tiles = (max_seqlen_q + BM - 1) / BM;
  prm.qscale = scale * kLog2e;

  // q as {D, Hq, T}: a box is 64 dims x 1 head x 128 query rows (swizzled).
  const uint64_t qdims[3] = {(uint64_t)head_dim, (uint64_t)num_q_heads, (uint64_t)total_q};
  const uint64_t qstr[2] = {(uint64_t)head_dim * 2, (uint64_t)num_q_heads * head_dim * 2};
  const uint32_t qbox[3] = {64u, 1u, (uint32_t)BM};
  // cache as {D, Hkv, block_size, NB}: a box is 64 dims x 1 head x 64 tokens x 1 block.
  const uint64_t kdims[4] = {(uint64_t)head_dim, (uint64_t)num_kv_heads, (uint64_t)block_size,
                             (uint64_t)num_blocks};
  const uint64_t kstr[3] = {(uint64_t)head_dim * 2, (uint64_t)num_kv_heads * head_dim * 2,
                            (uint64_t)block_size * num_kv_heads * head_dim * 2};
  const uint32_t kbox[4] = {64u, 1u, (uint32_t)BN, 1u};
  CUtensorMap tq, tk, tv;
  if (!encode_bf16_map(&tq, q, 3, qdims, qstr, qbox, true) ||
      !encode_bf16_map(&tk, k_cache, 4, kdims, kstr, kbox, true) ||
      !encode_bf16_map(&tv, v_cache, 4, kdims, kstr, kbox, true))
    return PKV_ERR_CUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool pair = (G % 2) == 0;
  if (head_dim == 128) return pair ? launch_prefill<128, 2>(tq, tk, tv, prm, st)
                                   : launch_prefill<128, 1>(tq, tk, tv, prm, st);
  return pair ? launch_prefill<64, 2>(tq, tk, tv, prm, st) : launch_prefill<64, 1>(tq, tk, tv, prm, st);
}
