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
//  * Persistent: one CTA per SM takes work units (sequence, 128-query tile,
//    pair of query heads of one GQA group) from an atomic counter in a small
//    caller workspace, in sequence-major order (sequences longest context
//    first, a sequence's heaviest tiles first, head groups innermost), so
//    that concurrent units reuse a sequence's K/V from L2 and the longest
//    units start first.  All roles run across unit boundaries: the next
//    unit's Q/K loads and first MMAs overlap this unit's last softmax and
//    epilogue.  The two heads of a unit share every K/V tile.
//  * Warp 0 fetches and decodes units (passing them to the other roles
//    through a small shared ring) and issues TMA for Q and K; warp 2 issues
//    TMA for V: 128B-swizzled 4-D boxes {64 dims, 1 head, 64 tokens, 1 block}
//    of 64-key tiles through the block table.
//  * Warp 1 issues S_h = Q_h K^T (tcgen05.mma, M=128, N=64, fp32 in tensor
//    memory, two buffers per head); warp 3 issues O_h += P_h V (M=128, N=D,
//    P from tensor memory, V MN-major).  Two issuers keep the tensor pipe
//    fed while either waits on a barrier.  For batches of short prompts the
//    kernel's other form gives each head its own issuer instead (warp 1:
//    head 0's S and P.V, warp 3: head 1's), so at the frequent unit
//    boundaries neither head waits on the other.  The four control warps take the
//    lowest warp ids: the schedulers favour them over the softmax warps
//    they share a sub-partition with (measured 1-3 % faster than placing
//    them after the softmax warps, 10 % faster than all four last).
//  * Warps 4.. (four per head, one per TMEM lane quarter, the two heads'
//    warps interleaved so each leads on two sub-partitions; one thread per
//    query row) read S, apply the causal mask offset by the cached length,
//    run the online softmax in fp32 (log2 domain; a row that sees the whole
//    key tile gets its max from the TMEM load itself, the load-with-max form
//    of tcgen05.ld that sm_103a adds), write P as bf16 over the S it came
//    from (half a tile at a time, each half's store in flight while the
//    next half's exponentials run), rescale O when the row max grows, and
//    finally normalise O and store bf16 rows.
#include <math.h>

#include "host_common.h"
#include "pkv_common.cuh"

namespace pkv {
namespace {

constexpr int BM = 128;  // query rows per tile (MMA M)
constexpr int BN = 64;   // keys per tile
constexpr int kUnitSlots = 4;  // depth of the shared ring of fetched units
constexpr int kMaxSorted = 256;  // sequences ordered longest-first in shared memory (more: as given)
constexpr int kPackMaxQ = 1024;  // longest prompt (new tokens) for which the packing kernel runs
constexpr int kPackMeanQ = 128;  // largest mean new tokens per sequence for it
constexpr int kPerHeadMeanQ = 1024;  // largest mean new tokens per sequence for one issuer per head
// Warp 0: unit fetcher + Q/K TMA producer; warp 1: S = QK^T MMA issuer;
// warp 2: V TMA producer; warp 3: P.V MMA issuer; then one 4-warp softmax
// group per head.
template <int NH>
constexpr int threads_for() { return 128 + 128 * NH; }
constexpr float kLog2e = 1.4426950408889634f;

// Caller workspace: the unit counter and the count of CTAs that finished
// fetching.  Zero between launches (the last CTA of each launch resets it).
struct PrefillWorkspace {
  unsigned int next_unit;
  unsigned int ctas_done;
};

struct PrefillParams {
  uint16_t *out;
  const int32_t *block_tables;
  const int32_t *cu_q;
  const int32_t *cu_k;
  int32_t *status;
  PrefillWorkspace *ws;
  int64_t num_blocks;
  int64_t total_q;
  int num_seqs;
  int sorted;        // num_seqs <= kMaxSorted: units follow the longest-first sequence order
  int num_q_heads;
  int num_kv_heads;
  int block_size;
  int max_blocks_per_seq;
  int q_tiles;       // ceil(max_seqlen_q / BM)
  unsigned int num_units;  // num_seqs * q_tiles * head groups
  float qscale;      // scale * log2(e)
  int out_32b;       // out is 32-byte aligned: rows are written with 256-bit stores
};

// 32-byte store of eight 32-bit words (address 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void *ptr, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(ptr), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// One work unit: query rows [q0, q0 + rows_valid) of sequence s, query heads
// h_first .. h_first + NH - 1, keys [0, n_kv * BN) of the sequence.
struct Unit {
  int s, q_begin, len_k, c, q0, rows_valid, n_kv, h_first, kvh;
  int pack;  // both heads' rows in one 128-row tile (rows_valid <= 64; packing kernels only)
};

// Unit index -> unit (sequence-major, heaviest tile of a sequence first, head
// groups innermost; sequences longest context first when `order` is in use).
// False when the index has no work (a tile past a short prompt) or its
// lengths are inconsistent (then PKV_DEV_BAD_SEQLEN is set).
template <int NH, bool kPack>
__device__ bool decode_unit(unsigned int idx, const PrefillParams &p, const uint32_t *order,
                            Unit &u) {
  const int HG = p.num_q_heads / NH;
  const int hg = (int)(idx % (unsigned)HG);
  idx /= (unsigned)HG;
  const int tr = (int)(idx % (unsigned)p.q_tiles);
  const int rank = (int)(idx / (unsigned)p.q_tiles);
  const int s = p.sorted ? 0xFFFF - (int)(order[rank] & 0xFFFFu) : rank;
  const int q_begin = p.cu_q[s];
  const int n = p.cu_q[s + 1] - q_begin;
  const int len_k = p.cu_k[s + 1] - p.cu_k[s];
  const int c = len_k - n;
  if (n <= 0) return false;
  const int ntq = (n + BM - 1) / BM;
  if (c < 0 || len_k > p.max_blocks_per_seq * p.block_size || ntq > p.q_tiles ||
      (int64_t)q_begin + n > p.total_q) {
    if (tr == 0 && hg == 0) flag_status(p.status, PKV_DEV_BAD_SEQLEN);
    if (c < 0 || len_k > p.max_blocks_per_seq * p.block_size || (int64_t)q_begin + n > p.total_q)
      return false;
  }
  const int t = ntq - 1 - tr;
  if (t < 0) return false;
  u.s = s;
  u.q_begin = q_begin;
  u.len_k = len_k;
  u.c = c;
  u.q0 = t * BM;
  u.rows_valid = min(BM, n - u.q0);
  u.n_kv = (min(len_k, c + u.q0 + u.rows_valid) + BN - 1) / BN;  // keys the tile needs
  u.h_first = hg * NH;
  u.kvh = u.h_first / (p.num_q_heads / p.num_kv_heads);
  u.pack = (kPack && NH == 2 && u.rows_valid <= BM / 2) ? 1 : 0;
  return true;
}

template <int D, int NH>
struct PrefillLayout {
  static constexpr int kQBytes = BM * D * 2;   // one head's Q tile
  static constexpr int kKVBytes = BN * D * 2;  // one K or V tile
  // Ring depths: the K/V slots that fit next to Q in 227 KiB of shared
  // memory (at most 12).  A K slot is held until its S MMAs finish, a V slot
  // until its P.V has run, so V gets the larger share.
  static constexpr int kSlots0 = (232448 - 3072 - NH * kQBytes) / kKVBytes;
  static constexpr int kSlots = kSlots0 < 12 ? kSlots0 : 12;
  static constexpr int kKStages = kSlots * 2 / 5;
  static constexpr int kVStages = kSlots - kKStages;
  static constexpr int q = 0;
  static constexpr int k = q + NH * kQBytes;
  static constexpr int v = k + kKStages * kKVBytes;
  static constexpr int bars = v + kVStages * kKVBytes;
  // barriers: q_full, q_empty, k_full[SK], v_full[SV], k_empty[SK], v_empty[SV],
  // s_full[NH][2], p_full[NH][2], p_free[NH][2], o_free[NH], unit_full[U],
  // unit_empty[U], drain
  static_assert(kKStages >= 2 && kVStages >= 2, "rings too shallow");
  static constexpr int kNumBars =
      2 + 2 * kKStages + 2 * kVStages + 7 * NH + 2 * kUnitSlots + 1;
  static constexpr int misc = bars + kNumBars * 8;  // tmem address, abort flag, unit ring
  static constexpr int ring = misc + 8;
  static constexpr int order = ring + (int)sizeof(Unit) * kUnitSlots;  // [kMaxSorted] sort keys
  static constexpr int total = order + 4 * kMaxSorted;
  static_assert(total + 1024 <= 232448, "shared memory");
  static constexpr int kCols = NH * D + 2 * NH * BN;  // per head: O and two S/P buffers
  static constexpr int kTmemCols = kCols <= 128 ? 128 : (kCols <= 256 ? 256 : 512);
};

// Tensor-memory columns (lane = query row): O_h (fp32) at kO + h*D, and two
// S buffers per head at kS + (2h + b)*BN, b = tile index & 1.  Tile g's S_h
// (fp32) goes to buffer g & 1; the softmax reads it into registers and
// writes P_h (bf16 pairs, the A operand of P.V) over its first BN/2 columns.
// So S of tile g + 1 is computed while the softmax of tile g runs, and S of
// tile g + 2 waits only for the P.V of tile g.
template <int D, int NH>
struct TmemCols {
  static constexpr uint32_t kO = 0;
  static constexpr uint32_t kS = NH * D;
};

// Paired fp32 arithmetic (one instruction for two lanes of a register pair):
// the same results as the scalar operations, half the instructions.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// Sequences longest context first (ties by index), so the longest units
// start first and the CTAs finish together.  Each sequence's key (key
// tiles << 16 | 0xFFFF - s) is unique; its place in the descending order is
// the number of larger keys, counted over the keys in shared memory: three
// CTA barriers, where the bitonic network this replaced took up to 36
// (measured: varlen prefill 494.1 -> 490.8 us, prefix-cached 74.2 -> 72.2
// us, mixed step 112.5 -> 110.3 us).  Inlined: out of line, the call made
// the kernel keep a larger stack frame and its loops ran 1.2 % slower.
// Every CTA sorts its own copy; all threads of the CTA call this.  The same
// pass prefetches cu_seqlens_q, which the first units read next.
static_assert(kMaxSorted <= threads_for<1>(), "one sort key per thread");
static __device__ __forceinline__ void sort_sequences(const PrefillParams &p, uint32_t *order) {
  const int n = p.num_seqs;  // <= kMaxSorted
  const int i = threadIdx.x;
  uint32_t key = 0;
  if (i < n) {
    if ((i & 31) == 0) asm volatile("prefetch.global.L1 [%0];" ::"l"(p.cu_q + i));
    const int lk = p.cu_k[i + 1] - p.cu_k[i];
    const uint32_t cost = lk <= 0 ? 0u : min((uint32_t)((lk + BN - 1) / BN), 0xFFFFu);
    key = (cost << 16) | (uint32_t)(0xFFFF - i);
    order[i] = key;
  }
  __syncthreads();
  int rank = 0;
  if (i < n)
    for (int x = 0; x < n; ++x) rank += order[x] > key ? 1 : 0;
  __syncthreads();
  if (i < n) order[rank] = key;
}

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
  const bool ok = mbar_wait_bounded(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// Barrier phases below count tiles (g) and units (iu) over the CTA's whole
// run, so they carry across unit boundaries.
template <int D, int NH, bool kPack, bool kPerHead>
__global__ void __launch_bounds__(threads_for<NH>(), 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_q64,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using L = PrefillLayout<D, NH>;
  constexpr int XR = D / 64;  // 128-byte swizzle regions across D
  constexpr int kKStages = L::kKStages;
  constexpr int kVStages = L::kVStages;
  constexpr uint32_t kOCol = TmemCols<D, NH>::kO;
  constexpr uint32_t kSCol = TmemCols<D, NH>::kS;
  constexpr int kKWarp = 0, kSWarp = 1, kVWarp = 2, kPVWarp = 3;  // then the softmax warps

  // ---- shared memory ----------------------------------------------------
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem + L::q;
  uint8_t *sK = smem + L::k;
  uint8_t *sV = smem + L::v;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bars);
  uint64_t *q_full = bars;
  uint64_t *q_empty = bars + 1;             // the unit's S MMAs no longer read Q
  uint64_t *k_full = bars + 2;
  uint64_t *v_full = k_full + kKStages;
  uint64_t *k_empty = v_full + kVStages;
  uint64_t *v_empty = k_empty + kKStages;
  uint64_t *s_full = v_empty + kVStages;    // [NH][2]: S in buffer b
  uint64_t *p_full = s_full + 2 * NH;       // [NH][2]: P written over it
  uint64_t *p_free = p_full + 2 * NH;       // [NH][2]: that P.V is done (O updated, buffer free)
  uint64_t *o_free = p_free + 2 * NH;       // [NH]: the epilogue has read O
  uint64_t *unit_full = o_free + NH;        // [kUnitSlots]
  uint64_t *unit_empty = unit_full + kUnitSlots;
  uint64_t *drain = unit_empty + kUnitSlots;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::misc + 4);
  Unit *unit_ring = reinterpret_cast<Unit *>(smem + L::ring);  // decoded units; s < 0 ends
  uint32_t *order = reinterpret_cast<uint32_t *>(smem + L::order);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    // Q, K and V slots are released by the S / P.V issuer, or by each head's
    // issuer when there is one per head.
    constexpr int kReleases = kPerHead ? NH : 1;
    mbar_init(q_empty, kReleases);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], kReleases);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], kReleases);
    }
    for (int h = 0; h < NH; ++h) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(&s_full[2 * h + b], 1);
        mbar_init(&p_full[2 * h + b], 128);  // the head's four softmax warps
        mbar_init(&p_free[2 * h + b], 1);
      }
      mbar_init(&o_free[h], 4);  // the 4 warps of the head's softmax group
    }
    // Unit ring readers: V producer, the MMA issuers, every softmax warp.
    constexpr int kIssuers = kPerHead ? NH : 2;
    for (int i = 0; i < kUnitSlots; ++i) {
      mbar_init(&unit_full[i], 1);
      mbar_init(&unit_empty[i], 1 + kIssuers + 4 * NH);
    }
    mbar_init(drain, kIssuers);  // one commit from each MMA issuer
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kSWarp) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  if (p.sorted) sort_sequences(p, order);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // The next unit from the ring (all readers see the same sequence).  False
  // at the end of the work or when the wait gives up.  Lane 0 of the calling
  // warp releases the slot.
  auto next_unit = [&](int &iu, Unit &u) -> bool {
    const int slot = iu % kUnitSlots;
    if (!warp_wait(&unit_full[slot], (iu / kUnitSlots) & 1, abort_flag)) return false;
    u = unit_ring[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&unit_empty[slot]);
    ++iu;
    return u.s >= 0;
  };

  if (warp == kKWarp || warp == kVWarp) {
    // ============ TMA producers: warp 0 fetches units and loads Q and K, ============
    // ============ warp 2 loads V                                          ============
    // The K and V rings turn over independently: a K slot is free once the
    // S MMAs that read it are done, a V slot once its P.V MMAs are done.
    const bool is_k = (warp == kKWarp);
    uint64_t *full = is_k ? k_full : v_full;
    uint64_t *empty = is_k ? k_empty : v_empty;
    uint8_t *ring = is_k ? sK : sV;
    const CUtensorMap *map = is_k ? &tm_k : &tm_v;
    const int nst = is_k ? kKStages : kVStages;
    int iu = 0, g = 0, q_loads = 0;
    bool ok = true;
    if (is_k && lane == 0) {
      tma_prefetch_map(&tm_q);
      if (kPack) tma_prefetch_map(&tm_q64);
      tma_prefetch_map(&tm_k);
    } else if (lane == 0) {
      tma_prefetch_map(&tm_v);
    }
    for (;;) {
      Unit u;
      bool have;
      if (is_k) {
        // Fetch and decode the next unit with work and publish it to the
        // ring, so the other roles start a unit without reading the
        // sequence lengths themselves.  A unit without work means the rest of
        // its sequence's units have none either (later tiles, or an empty or
        // inconsistent sequence): move the shared counter to the next
        // sequence instead of taking them one by one.
        have = false;
        if (lane == 0) {
          const unsigned int per_seq = (unsigned)(p.q_tiles * (p.num_q_heads / NH));
          for (;;) {
            const unsigned int i = atomicAdd(&p.ws->next_unit, 1u);
            if (i >= p.num_units) break;
            if (decode_unit<NH, kPack>(i, p, order, u)) {
              have = true;
              break;
            }
            atomicMax(&p.ws->next_unit, (i / per_seq + 1) * per_seq);
          }
          if (!have) u.s = -1;
        }
        const int slot = iu % kUnitSlots;
        if (iu >= kUnitSlots)
          ok = warp_wait(&unit_empty[slot], ((iu / kUnitSlots) - 1) & 1, abort_flag);
        if (!ok) break;
        if (lane == 0) {
          unit_ring[slot] = u;
          mbar_arrive(&unit_full[slot]);  // (release: orders the stores above)
        }
        ++iu;
        have = __shfl_sync(0xffffffffu, have ? 1 : 0, 0) != 0;
        if (!have) break;
      } else {
        have = next_unit(iu, u);
      }
      if (!have) break;
      if (lane == 0) {  // (only lane 0 of warp 0 holds the decoded unit)
        if (is_k) {
          // Q of this unit once the previous unit's S MMAs are done with Q.
          if (iu >= 2) ok = mbar_wait_bounded(q_empty, (iu - 2) & 1, abort_flag);
          if (ok && kPack && u.pack) {
            // Packed unit: each head's first 64 query rows, head h in rows
            // 64h .. 64h + 63 of the first head's Q tile.
            ++q_loads;
            mbar_arrive_expect_tx(q_full, NH * L::kQBytes / 2);
            for (int h = 0; h < NH; ++h)
              for (int x = 0; x < XR; ++x)
                tma_load_3d(sQ + x * BM * 128 + h * (BM / 2) * 128, &tm_q64, q_full, x * 64,
                            u.h_first + h, u.q_begin + u.q0);
          } else if (ok) {
            ++q_loads;
            mbar_arrive_expect_tx(q_full, NH * L::kQBytes);
            for (int h = 0; h < NH; ++h)
              for (int x = 0; x < XR; ++x)
                tma_load_3d(sQ + h * L::kQBytes + x * BM * 128, &tm_q, q_full, x * 64,
                            u.h_first + h, u.q_begin + u.q0);
          }
        }
        for (int jt = 0; jt < u.n_kv && ok; ++jt, ++g) {
          const int st = g % nst;
          if (g >= nst && !mbar_wait_bounded(&empty[st], ((g / nst) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const int key0 = jt * BN;
          const int lb = key0 / p.block_size;
          const int off = key0 - lb * p.block_size;
          int blk = p.block_tables[(int64_t)u.s * p.max_blocks_per_seq + lb];
          if (blk < 0 || (int64_t)blk >= p.num_blocks) {
            flag_status(p.status, PKV_DEV_BAD_BLOCK);
            blk = 0;
          }
          mbar_arrive_expect_tx(&full[st], L::kKVBytes);
          for (int x = 0; x < XR; ++x)
            tma_load_4d(ring + st * L::kKVBytes + x * BN * 128, map, &full[st], x * 64, u.kvh,
                        off, blk);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      g = __shfl_sync(0xffffffffu, g, 0);
      if (!ok) break;
    }
    if (lane == 0) {
      // Do not leave while copies into this CTA's shared memory are in flight.
      if (is_k && q_loads > 0 && !mbar_wait_bounded(q_full, (q_loads - 1) & 1, nullptr))
        flag_status(p.status, PKV_DEV_TIMEOUT);
      for (int i = max(0, g - nst); i < g; ++i)
        if (!mbar_wait_bounded(&full[i % nst], (i / nst) & 1, nullptr))
          flag_status(p.status, PKV_DEV_TIMEOUT);
      if (is_k) {
        // This CTA fetches no more units; the last CTA to get here leaves the
        // workspace zeroed for the next launch.
        __threadfence();
        if (atomicAdd(&p.ws->ctas_done, 1u) == gridDim.x - 1) {
          p.ws->next_unit = 0;
          p.ws->ctas_done = 0;
          __threadfence();
        }
      }
    }
  } else if (warp == kSWarp || warp == kPVWarp) {
    if constexpr (kPerHead) {
      // ============ MMA issuers, one per head: warp 1 head 0, warp 3 head 1 ============
      // Each issues its head's S = Q K^T for a tile, then the P.V of the tile
      // before it, so neither head waits on the other's barriers.  A K or V
      // slot (and Q) is free once both heads are done with it.  Shared-memory
      // matrix descriptors are built once; an MMA only adds the operand's
      // offset to the address field (bits 0-13, bytes / 16).
      const int h = warp == kSWarp ? 0 : 1;
      if (h < NH) {
        constexpr uint32_t idesc_s = umma_idesc_bf16(BM, BN, false, false);
        constexpr uint32_t idesc_o = umma_idesc_bf16(BM, D, false, true);
        const uint64_t dq = umma_desc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dk = umma_desc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t dv = umma_desc_sw128(smem_u32(sV), BN * 128, 1024);
        // g: tiles of every unit (ring slots); gh, uh: this head's tiles and
        // units (packing kernels: head 1 takes no part in packed units).
        int iu = 0, g = 0, gh = 0, uh = 0;
        bool ok = true;
        Unit u;
        // The P.V of this head's previous tile: ring tile, head tile, head unit.
        bool pend = false, pfirst = false;
        int pg = 0, pgh = 0, puh = 0;
        // O_h += P_h V once V is in and the head's P is written; then the S/P
        // buffer and the V slot are released.  A unit's first P.V overwrites
        // O_h, so it also waits until the previous unit's epilogue has read O_h.
        auto issue_pv = [&]() -> bool {
          const int pst = pg % kVStages;
          if (!mbar_wait_bounded(&v_full[pst], (pg / kVStages) & 1, abort_flag)) return false;
          if (!mbar_wait_bounded(&p_full[2 * h + (pgh & 1)], (pgh >> 1) & 1, abort_flag))
            return false;
          if (pfirst && puh >= 1 && !mbar_wait_bounded(&o_free[h], (puh - 1) & 1, abort_flag))
            return false;
          tc_fence_after_sync();
          const uint64_t dv_st = dv + (uint64_t)((pst * L::kKVBytes) >> 4);
          const uint32_t pa = tmem + kSCol + (2 * h + (pgh & 1)) * BN;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            umma_bf16_tmem_a(tmem + kOCol + h * D, pa + kk * 8,
                             dv_st + (uint64_t)((kk * 16 * 128) >> 4), idesc_o,
                             (!pfirst || kk > 0) ? 1u : 0u);
          umma_commit(&p_free[2 * h + (pgh & 1)]);
          umma_commit(&v_empty[pst]);
          return true;
        };
        while (ok && next_unit(iu, u)) {
          const bool pk = kPack && u.pack;
          if (lane == 0) {
            ok = mbar_wait_bounded(q_full, (iu - 1) & 1, abort_flag);
            if (pk && h == 1) {
              // A packed unit has one S and one P.V (both heads' rows, head 0's
              // tensor memory): this head issues its pending P.V, then only
              // releases the unit's Q and each K and V slot once it has been
              // filled, tile by tile (head 0's S and P.V need the rings to turn).
              if (ok && pend) {
                ok = issue_pv();
                pend = false;
              }
              for (int jt = 0; jt < u.n_kv && ok; ++jt) {
                const int gg = g + jt;
                ok = mbar_wait_bounded(&k_full[gg % kKStages], (gg / kKStages) & 1, abort_flag);
                if (ok) mbar_arrive(&k_empty[gg % kKStages]);
                if (ok)
                  ok = mbar_wait_bounded(&v_full[gg % kVStages], (gg / kVStages) & 1, abort_flag);
                if (ok) mbar_arrive(&v_empty[gg % kVStages]);
              }
              if (ok) mbar_arrive(q_empty);
            } else {
              // S_h into buffer gh & 1 once K is in and the P.V two head tiles
              // back (which read P from that buffer) is done.
              for (int jt = 0; jt < u.n_kv && ok; ++jt) {
                const int gg = g + jt, gq = gh + jt;
                const int st = gg % kKStages;
                const int b = gq & 1;
                ok = mbar_wait_bounded(&k_full[st], (gg / kKStages) & 1, abort_flag);
                if (ok && gq >= 2)
                  ok = mbar_wait_bounded(&p_free[2 * h + b], ((gq - 2) >> 1) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after_sync();
                const uint64_t dk_st = dk + (uint64_t)((st * L::kKVBytes) >> 4);
                const uint32_t d = tmem + kSCol + (2 * h + b) * BN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                  const uint32_t off = (kk & 3) * 32;
                  umma_bf16(d, dq + (uint64_t)((h * L::kQBytes + (kk / 4) * BM * 128 + off) >> 4),
                            dk_st + (uint64_t)(((kk / 4) * BN * 128 + off) >> 4), idesc_s,
                            kk > 0 ? 1u : 0u);
                }
                umma_commit(&s_full[2 * h + b]);
                umma_commit(&k_empty[st]);
                if (jt == u.n_kv - 1) umma_commit(q_empty);
                if (pend) {
                  ok = issue_pv();
                  if (!ok) break;
                }
                pend = true;
                pfirst = jt == 0;
                pg = gg;
                pgh = gq;
                puh = uh;
              }
            }
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          g += u.n_kv;
          if (!(pk && h == 1)) {
            gh += u.n_kv;
            ++uh;
          }
        }
        if (lane == 0) {
          if (ok && pend) ok = issue_pv();
          // Wait for this issuer's MMAs before tensor memory is freed.
          umma_commit(drain);
          if (!mbar_wait_bounded(drain, 0, nullptr)) flag_status(p.status, PKV_DEV_TIMEOUT);
        }
      }
    } else {
      // ============ MMA issuers: warp 1 issues S = QK^T, warp 3 O += PV ============
      // Two issuing threads keep the tensor pipe fed while either one waits on
      // a barrier (its queue of issued MMAs is short).  Shared-memory matrix
      // descriptors are built once; an MMA only adds the operand's offset to
      // the address field (bits 0-13, bytes / 16).
      int iu = 0, g = 0;
      // Packing kernels: head 1 takes no part in packed units, so its S/P
      // buffers and O count their own tiles (g1) and units (u1).
      int g1 = 0, u1 = 0;
      bool ok = true;
      Unit u;
      if (warp == kSWarp) {
        constexpr uint32_t idesc_s = umma_idesc_bf16(BM, BN, false, false);
        const uint64_t dq = umma_desc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dk = umma_desc_sw128(smem_u32(sK), 16, 1024);
        while (ok && next_unit(iu, u)) {
          const bool pk = kPack && u.pack;
          if (lane == 0) {
            ok = mbar_wait_bounded(q_full, (iu - 1) & 1, abort_flag);
            // Per tile: S_h for every head into buffer g & 1 once K is in
            // and the P.V two tiles back (which read P from that buffer) is done.
            // A packed unit has one 128-row S (both heads' rows) in head 0's buffers.
            for (int jt = 0; jt < u.n_kv && ok; ++jt, ++g) {
              const int st = g % kKStages;
              ok = mbar_wait_bounded(&k_full[st], (g / kKStages) & 1, abort_flag);
              const uint64_t dk_st = dk + (uint64_t)((st * L::kKVBytes) >> 4);
#pragma unroll
              for (int h = 0; h < NH && ok; ++h) {
                if (pk && h > 0) break;
                const int gh = (kPack && h == 1) ? g1 + jt : g;  // head h's tile count
                const int b = gh & 1;
                if (gh >= 2)
                  ok = mbar_wait_bounded(&p_free[2 * h + b], ((gh - 2) >> 1) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t d = tmem + kSCol + (2 * h + b) * BN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                  const uint32_t off = (kk & 3) * 32;
                  umma_bf16(d, dq + (uint64_t)((h * L::kQBytes + (kk / 4) * BM * 128 + off) >> 4),
                            dk_st + (uint64_t)(((kk / 4) * BN * 128 + off) >> 4), idesc_s,
                            kk > 0 ? 1u : 0u);
                }
                umma_commit(&s_full[2 * h + b]);
              }
              if (ok) umma_commit(&k_empty[st]);
            }
            if (ok) umma_commit(q_empty);
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          g = __shfl_sync(0xffffffffu, g, 0);
          if (kPack && !pk) g1 += u.n_kv;
        }
      } else {
        constexpr uint32_t idesc_o = umma_idesc_bf16(BM, D, false, true);
        const uint64_t dv = umma_desc_sw128(smem_u32(sV), BN * 128, 1024);
        while (ok && next_unit(iu, u)) {
          const bool pk = kPack && u.pack;
          if (lane == 0) {
            // Per tile, in head order: O_h += P_h V (P from tensor memory) once V
            // is in and the head's P is written; then the S/P buffer and the V
            // slot are released.  A unit's first P.V overwrites O_h, so it also
            // waits until the previous unit's epilogue has read O_h.  Head order
            // keeps every head's last P.V behind head 0's softmax warps, which clear the V
            // rows past the context before it publishes its P.  A packed unit
            // has one P.V (both heads' rows) into head 0's O.
            for (int jt = 0; jt < u.n_kv && ok; ++jt, ++g) {
              const int pst = g % kVStages;
              ok = mbar_wait_bounded(&v_full[pst], (g / kVStages) & 1, abort_flag);
              const uint64_t dv_st = dv + (uint64_t)((pst * L::kKVBytes) >> 4);
#pragma unroll
              for (int h = 0; h < NH && ok; ++h) {
                if (pk && h > 0) break;
                const int gh = (kPack && h == 1) ? g1 + jt : g;  // head h's tile count
                const int uh = (kPack && h == 1) ? u1 : iu - 1;  // head h's units before this one
                ok = mbar_wait_bounded(&p_full[2 * h + (gh & 1)], (gh >> 1) & 1, abort_flag);
                if (ok && jt == 0 && uh >= 1)
                  ok = mbar_wait_bounded(&o_free[h], (uh - 1) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t pa = tmem + kSCol + (2 * h + (gh & 1)) * BN;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                  umma_bf16_tmem_a(tmem + kOCol + h * D, pa + kk * 8,
                                   dv_st + (uint64_t)((kk * 16 * 128) >> 4), idesc_o,
                                   (jt > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&p_free[2 * h + (gh & 1)]);
              }
              if (ok) umma_commit(&v_empty[pst]);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          g = __shfl_sync(0xffffffffu, g, 0);
          if (kPack && !pk) {
            g1 += u.n_kv;
            ++u1;
          }
        }
      }
      if (lane == 0) {
        // Wait for the MMAs of both issuers before tensor memory is freed.
        umma_commit(drain);
        if (!mbar_wait_bounded(drain, 0, nullptr)) flag_status(p.status, PKV_DEV_TIMEOUT);
      }
    }
  } else {
    // ================= softmax / epilogue: four warps per head ==================
    // The head this warp serves.  Each head needs one warp per TMEM lane
    // quarter (warp & 3); with two heads, warps 4, 5, 10, 11 serve head 0 and
    // 6, 7, 8, 9 head 1, so that on two of the four SM sub-partitions each
    // head's warp has the lower warp id (issue priority) and neither head
    // trails the other (measured: varlen prefill 497.8 -> 494.8 us, prefix
    // 79.3 -> 78.4 us, against warps 4-7 / 8-11).
    const int h = NH == 2 ? ((((warp - 4) >> 1) ^ ((warp - 4) >> 2)) & 1) : 0;
    const int quarter = warp & 3;   // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float qs = p.qscale;
    int iu = 0, g = 0;
    // Packing kernels: head 1's warps take no part in packed units; its S/P
    // buffer barriers count only the tiles it processes (g1).
    int g1 = 0;
    bool ok = true;
    Unit u;
    // Epilogue of a unit (rows from query row e_row0, e_rows of them valid,
    // heads from e_h): O / l -> bf16 rows once its last P.V (tile g_last) is
    // in O.  Run after the next unit's first P is published, so the wait for
    // that P.V overlaps the first softmax tile of the next unit.  Waited for
    // through g_last's buffer barrier: its use before (tile g_last - 2) was
    // done before S of g_last was computed, and its next use needs a P this
    // head's warps have not yet written, so the parity wait cannot alias.
    // In a packed unit (head 0's warps only) row r holds query row r % 64 of
    // head e_h + r / 64.
    auto epilogue = [&](int e_row0, int e_rows, int e_h, float l_e, int g_last,
                        bool e_pack) -> bool {
      if (!warp_wait(&p_free[2 * h + (g_last & 1)], (g_last >> 1) & 1, abort_flag)) return false;
      tc_fence_after_sync();
      const float inv = 1.f / l_e;
      const int orow = (kPack && e_pack) ? (row & (BM / 2 - 1)) : row;
      const int ohead = (kPack && e_pack) ? (row >> 6) : h;
      uint16_t *dst = p.out + ((int64_t)(e_row0 + orow) * p.num_q_heads + e_h + ohead) * D;
#pragma unroll 1
      for (int half = 0; half < D / 64; ++half) {
        float ov[64];
        tmem_load64(tmem + lane_base + kOCol + h * D + half * 64, ov);
        if (orow < e_rows) {
#pragma unroll
          for (int i = 0; i < 64; i += 16) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float2 o2 = mul2(make_float2(ov[i + 2 * e], ov[i + 2 * e + 1]), make_float2(inv, inv));
              w[e] = pack_bf16x2(o2.x, o2.y);
            }
            if (p.out_32b) {
              st_global_v8(dst + half * 64 + i, w);
            } else {
              *reinterpret_cast<uint4 *>(dst + half * 64 + i) = make_uint4(w[0], w[1], w[2], w[3]);
              *reinterpret_cast<uint4 *>(dst + half * 64 + i + 8) = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
        }
      }
      // O is read: the next unit's first P.V may overwrite it.
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[h]);
      return true;
    };
    bool pending = false;  // a unit's epilogue is still to run
    int e_row0 = 0, e_rows = 0, e_h = 0, e_g = 0;
    bool e_pack = false;
    float e_l = 0.f;
    while (ok && next_unit(iu, u)) {
      const bool pk = kPack && u.pack;
      if (pk && h == 1) {  // a packed unit has no work for the second head's warps
        if (pending) {
          pending = false;
          ok = epilogue(e_row0, e_rows, e_h, e_l, e_g, e_pack);
        }
        g += u.n_kv;
        continue;
      }
      const int prow = pk ? (row & (BM / 2 - 1)) : row;  // the row's query index in the tile
      const int key_limit = min(u.c + u.q0 + prow, u.len_k - 1);  // last key this row may see
      // Running max in log2 units.  It is only raised (and O rescaled) when a
      // tile's max exceeds it by more than 8, so P stays <= 2^8; l and O share
      // the same reference, so the final O / l is unchanged.
      float m_ref = -INFINITY;
      float l_run = 0.f;
      for (int jt = 0; jt < u.n_kv && ok; ++jt, ++g) {
        const int key0 = jt * BN;
        const int gt = (kPack && h == 1) ? g1 + jt : g;  // this head's S/P buffer turns
        const uint32_t sp = tmem + lane_base + kSCol + (2 * h + (gt & 1)) * BN;  // S, then P
        ok = warp_wait(&s_full[2 * h + (gt & 1)], (gt >> 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after_sync();
        float sv[BN];
        static_assert(BN == 64, "S is read with one 64-column TMEM load");
        float alpha = 1.f;
        float rs = 0.f;
        // A warp whose 32 query rows all lie past the tile's valid rows (a
        // decode row, a prompt's ragged last tile) skips the arithmetic and
        // the P store: those rows' outputs are never written, and P of a row
        // only reaches that row of O.  It still takes part in every barrier.
        const bool live = (pk ? ((quarter * 32) & (BM / 2 - 1)) : quarter * 32) < u.rows_valid;
        if (live) {
          // Tile max of the scaled logits over this row's visible keys: for a
          // row that sees the whole tile it comes with the TMEM load.
          const bool full_row = key0 + BN - 1 <= key_limit;
          float mt;
          {
            float e0 = -INFINITY;
            if (qs > 0.f) {
              float vmax;
              tmem_load64_max(sp, sv, vmax);
              if (full_row) {
                e0 = vmax;
              } else {
                // Keys past the row's limit become -inf (their P is then
                // exactly 0 in the unmasked exponential loop below).
                const int nvis = key_limit - key0;
                float e1 = -INFINITY, e2 = -INFINITY, e3 = -INFINITY;
#pragma unroll
                for (int i = 0; i < BN; i += 4) {
                  sv[i] = i <= nvis ? sv[i] : -INFINITY;
                  sv[i + 1] = i + 1 <= nvis ? sv[i + 1] : -INFINITY;
                  sv[i + 2] = i + 2 <= nvis ? sv[i + 2] : -INFINITY;
                  sv[i + 3] = i + 3 <= nvis ? sv[i + 3] : -INFINITY;
                  e0 = fmaxf(e0, sv[i]);
                  e1 = fmaxf(e1, sv[i + 1]);
                  e2 = fmaxf(e2, sv[i + 2]);
                  e3 = fmaxf(e3, sv[i + 3]);
                }
                e0 = fmaxf(fmaxf(e0, e1), fmaxf(e2, e3));
              }
              mt = e0 * qs;
            } else {
              tmem_load64(sp, sv);
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
          if (jt == 0 || mt > m_ref + 8.f) {
            const float m_new = fmaxf(m_ref, mt);
            alpha = (m_ref == -INFINITY) ? 0.f : fast_exp2(m_ref - m_new);
            m_ref = m_new;
          }
          {
            // Exponentials in two halves of the tile; each half's P (bf16
            // pairs, over the first half of this tile's S buffer) is stored
            // while the next half is computed.
            const float2 q2 = make_float2(qs, qs), nm2 = make_float2(-m_ref, -m_ref);
            float2 r01 = make_float2(0.f, 0.f), r23 = make_float2(0.f, 0.f);
            const bool dense = full_row || qs > 0.f;  // no mask to apply in the loop
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              if (dense) {
#pragma unroll
                for (int i = hf * (BN / 2); i < (hf + 1) * (BN / 2); i += 4) {
                  const float2 x01 = fma2(make_float2(sv[i], sv[i + 1]), q2, nm2);
                  const float2 x23 = fma2(make_float2(sv[i + 2], sv[i + 3]), q2, nm2);
                  sv[i] = fast_exp2(x01.x);
                  sv[i + 1] = fast_exp2(x01.y);
                  sv[i + 2] = fast_exp2(x23.x);
                  sv[i + 3] = fast_exp2(x23.y);
                  r01 = add2(r01, make_float2(sv[i], sv[i + 1]));
                  r23 = add2(r23, make_float2(sv[i + 2], sv[i + 3]));
                }
              } else {
#pragma unroll
                for (int i = hf * (BN / 2); i < (hf + 1) * (BN / 2); i += 4) {
#pragma unroll
                  for (int w = 0; w < 4; ++w)
                    sv[i + w] =
                        (key0 + i + w <= key_limit) ? fast_exp2(fmaf(sv[i + w], qs, -m_ref)) : 0.f;
                  r01 = add2(r01, make_float2(sv[i], sv[i + 1]));
                  r23 = add2(r23, make_float2(sv[i + 2], sv[i + 3]));
                }
              }
              float pw[BN / 4];
#pragma unroll
              for (int i = 0; i < BN / 4; ++i)
                pw[i] = __uint_as_float(
                    pack_bf16x2(sv[hf * (BN / 2) + 2 * i], sv[hf * (BN / 2) + 2 * i + 1]));
              tmem_store16_async(sp + hf * (BN / 4), pw);
            }
            tmem_wait_st();
            rs = (r01.x + r01.y) + (r23.x + r23.y);
          }
        }
        if (live && jt > 0 && __any_sync(0xffffffffu, alpha < 1.f)) {
          // O is rescaled once the previous P.V has landed in it (the next
          // waits for this tile's P).  Waited for through that tile's buffer:
          // its use before (tile g - 3) was done before S of tile g - 1 was
          // computed, and its next use needs this tile's P, so the parity
          // wait cannot alias.
          ok = warp_wait(&p_free[2 * h + ((gt - 1) & 1)], ((gt - 1) >> 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after_sync();
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            float ov[32];
            const uint32_t oa = tmem + lane_base + kOCol + h * D + cc * 32;
            tmem_load32(oa, ov);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 o2 = mul2(make_float2(ov[i], ov[i + 1]), make_float2(alpha, alpha));
              ov[i] = o2.x;
              ov[i + 1] = o2.y;
            }
            tmem_store32(oa, ov);
          }
        }
        l_run = l_run * alpha + rs;
        if ((kPerHead || h == 0) && key0 + BN > u.len_k) {
          // Keys past the context may hold stale bits (even NaN); P is zero
          // there, but 0 * NaN is not, so clear those V rows first.  (Every
          // head's last P.V is issued after these warps' arrival.)
          ok = warp_wait(&v_full[g % kVStages], (g / kVStages) & 1, abort_flag);
          if (!ok) break;
          const int first = u.len_k - key0;
          uint8_t *vt = sV + (g % kVStages) * L::kKVBytes;
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
        tc_fence_before_sync();
        mbar_arrive(&p_full[2 * h + (gt & 1)]);
        if (pending) {  // the previous unit's epilogue, after this unit's first P
          pending = false;
          ok = epilogue(e_row0, e_rows, e_h, e_l, e_g, e_pack);
        }
      }
      if (!ok) break;
      pending = true;
      e_row0 = u.q_begin + u.q0;
      e_rows = u.rows_valid;
      e_h = u.h_first;
      e_l = l_run;
      e_g = ((kPack && h == 1) ? g1 + u.n_kv : g) - 1;
      e_pack = pk;
      if (kPack && h == 1) g1 += u.n_kv;
    }
    if (ok && pending) ok = epilogue(e_row0, e_rows, e_h, e_l, e_g, e_pack);
    tc_fence_before_sync();
  }

  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) flag_status(p.status, PKV_DEV_TIMEOUT);
  if (warp == kSWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int D, int NH, bool kPack, bool kPerHead>
pkv_status launch_prefill(const CUtensorMap &tq, const CUtensorMap &tq64, const CUtensorMap &tk,
                          const CUtensorMap &tv, const PrefillParams &prm, cudaStream_t stream) {
  using L = PrefillLayout<D, NH>;
  int smem = L::total + 1024;
  // Resident CTAs per SM must not ask for more than 512 TMEM columns in
  // total, or tcgen05.alloc would stall: pad shared memory to cap occupancy.
  const int max_ctas = 512 / L::kTmemCols;
  const int per_sm = 228 * 1024;
  const int min_bytes = per_sm / (max_ctas + 1) + 1;
  if (smem < min_bytes) smem = min_bytes;
  int resident = 0;
  if (!kernel_smem_setup((const void *)paged_prefill_kernel<D, NH, kPack, kPerHead>,
                         threads_for<NH>(), smem, &resident))
    return PKV_ERR_CUDA;
  // Persistent: as many CTAs as can be resident, no more than there are units.
  const int ctas_per_sm = resident < max_ctas ? resident : max_ctas;
  int64_t grid = (int64_t)device_sm_count() * ctas_per_sm;
  if (grid > (int64_t)prm.num_units) grid = prm.num_units;
  if (grid < 1) grid = 1;
  paged_prefill_kernel<D, NH, kPack, kPerHead>
      <<<(unsigned)grid, threads_for<NH>(), smem, stream>>>(tq, tq64, tk, tv, prm);
  return launch_status();
}

}  // namespace
}  // namespace pkv

extern "C" size_t pkv_prefill_workspace_size(void) { return 256; }

extern "C" pkv_status pkv_paged_prefill_attn(uint16_t *out, const uint16_t *q,
                                             const uint16_t *k_cache, const uint16_t *v_cache,
                                             const int32_t *block_tables,
                                             const int32_t *cu_seqlens_q,
                                             const int32_t *cu_seqlens_k, int num_seqs,
                                             int64_t total_q, int max_seqlen_q, int num_q_heads,
                                             int num_kv_heads, int head_dim, int block_size,
                                             int max_blocks_per_seq, int64_t num_blocks,
                                             float scale, void *workspace,
                                             size_t workspace_bytes, int32_t *dev_status,
                                             void *stream) {
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
  if (!isfinite(scale)) return PKV_ERR_INVALID_ARG;  // NaN or infinite
  if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0) return PKV_OK;
  if (total_q > 0x7FFFFFFFLL) return PKV_ERR_UNSUPPORTED;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !cu_seqlens_q || !cu_seqlens_k)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < pkv_prefill_workspace_size() ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return PKV_ERR_WORKSPACE;

  const bool two_heads = (G % 2) == 0;  // a CTA serves two query heads of one group
  const int64_t q_tiles = (max_seqlen_q + BM - 1) / BM;
  const int64_t units = q_tiles * num_seqs * (num_q_heads / (two_heads ? 2 : 1));
  if (units > 0x7FFFFFFFLL) return PKV_ERR_UNSUPPORTED;

  PrefillParams prm;
  prm.out = out;
  prm.block_tables = block_tables;
  prm.cu_q = cu_seqlens_q;
  prm.cu_k = cu_seqlens_k;
  prm.status = dev_status;
  prm.ws = static_cast<PrefillWorkspace *>(workspace);
  prm.num_blocks = num_blocks;
  prm.total_q = total_q;
  prm.num_seqs = num_seqs;
  prm.sorted = num_seqs <= kMaxSorted ? 1 : 0;
  prm.num_q_heads = num_q_heads;
  prm.num_kv_heads = num_kv_heads;
  prm.block_size = block_size;
  prm.max_blocks_per_seq = max_blocks_per_seq;
  prm.q_tiles = (int)q_tiles;
  prm.num_units = (unsigned int)units;
  prm.qscale = scale * kLog2e;
  prm.out_32b = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0;

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
  // Decode-heavy batches (at most kPackMeanQ new tokens per sequence on
  // average, none over kPackMaxQ) run the packing kernel: its query tiles
  // with at most 64 valid rows (decode rows, short prompts, ragged last
  // tiles) hold both heads of the pair, 64 rows each, in one 128-row MMA
  // tile (one S and one P.V per key tile instead of two).  Measured: the
  // mixed step (48 decode rows + 8 chunks) 117.6 -> 112.7 us; on the
  // prefix-cached batch (19 % of its work packable) the packing kernel's
  // other units ran slower and the whole call went 78.4 -> 81.2 us, so
  // batches like it keep the kernel without the path.
  const bool pack = two_heads && max_seqlen_q <= kPackMaxQ &&
                    total_q <= (int64_t)kPackMeanQ * num_seqs;
  // Batches of short prompts (mean new tokens per sequence at most
  // kPerHeadMeanQ: many short units, so many unit boundaries) run one MMA
  // issuer per head, so neither head waits on the other's barriers at a
  // boundary.  Measured: prefix-cached batch 78.5 -> 74.8 us; the varlen
  // prefill (long prompts) 495.4 -> 501.8 us and the mixed step 112.6 ->
  // 113.8 us with it, so those keep one S issuer and one P.V issuer.
  const bool per_head = two_heads && !pack && total_q <= (int64_t)kPerHeadMeanQ * num_seqs;
  const uint32_t qbox64[3] = {64u, 1u, (uint32_t)(BM / 2)};
  CUtensorMap tq, tq64, tk, tv;
  if (pack && !encode_bf16_map(&tq64, q, 3, qdims, qstr, qbox64, true)) return PKV_ERR_CUDA;
  if (!encode_bf16_map(&tq, q, 3, qdims, qstr, qbox, true) ||
      !encode_bf16_map(&tk, k_cache, 4, kdims, kstr, kbox, true) ||
      !encode_bf16_map(&tv, v_cache, 4, kdims, kstr, kbox, true))
    return PKV_ERR_CUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!pack) tq64 = tq;  // (not read)
  if (head_dim == 128) {
    if (!two_heads) return launch_prefill<128, 1, false, false>(tq, tq64, tk, tv, prm, st);
    if (pack) return launch_prefill<128, 2, true, false>(tq, tq64, tk, tv, prm, st);
    return per_head ? launch_prefill<128, 2, false, true>(tq, tq64, tk, tv, prm, st)
                    : launch_prefill<128, 2, false, false>(tq, tq64, tk, tv, prm, st);
  }
  if (!two_heads) return launch_prefill<64, 1, false, false>(tq, tq64, tk, tv, prm, st);
  if (pack) return launch_prefill<64, 2, true, false>(tq, tq64, tk, tv, prm, st);
  return per_head ? launch_prefill<64, 2, false, true>(tq, tq64, tk, tv, prm, st)
                  : launch_prefill<64, 2, false, false>(tq, tq64, tk, tv, prm, st);
}
