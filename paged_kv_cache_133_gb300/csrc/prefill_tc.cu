// Ragged causal prefill on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Query token i of a sequence with c cached tokens sits at position c + i and
// sees keys 0 .. c + i of its own sequence (bottom-right aligned causal mask;
// "vLLM 原理" §3.7: new queries attend to the whole cached sequence).  Keys
// are consumed in tiles of 128 positions; each tile is gathered from the
// paged cache by TMA, one box per physical block found through the sequence's
// block table ("vLLM Continuous Batching：从 Forward Shape 理解两个核心参数"
// §2.3补充 第二步).
//
// Work item: 128 query tokens of one sequence for TWO query heads A and B of
// the same kv head (so every K/V tile feeds both), or one head when the group
// has an odd head left over.  An item's cost is its number of 128-key tiles;
// token tile t of a sequence with c cached tokens has cost ceil(c/128) + t + 1
// (one less for a short last tile).  Items are listed by that level,
// highest first, so the list is sorted by cost.  The grid is persistent (one
// CTA per SM): CTA b starts with item b, and then a scheduler warp in each
// CTA takes the next item number from a global counter (atomicAdd) whenever
// its CTA has room, so CTAs that drew cheap items draw more and all finish
// together.  The numbers cover existing items only (each CTA tabulates the
// items per level in shared memory and maps a number to its item), so no draw
// comes back empty.
//
// A token tile of at most 64 tokens (the tail of a chunk) is "packed" when
// the group splits into fours: each side's 128 rows hold two heads (rows
// 0-63 one head, 64-127 the next), so one item covers four heads with half
// the products.  A third mode (kCasc) runs the prefix pass of a shared-prefix
// decode: a side's rows are the (decode token, query head) pairs of a kv
// head, keys are a chunk of the shared prefix with no causal mask, and the
// epilogue writes fp32 partials (O, m, l) for the split combine.
//
// Warp roles (512 threads, four warpgroups):
//   warps 0-3   softmax of tile A (thread r = query row r = TMEM lane r)
//   warps 4-7   softmax of tile B
//   warp 8      TMA producer of K_j (2-stage ring)
//   warp 9      TMEM allocation and MMA issue (one lane)
//   warp 10     TMA producer of V_j (2-stage ring)
//   warp 11     scheduler: draws items from the global queue, hands them to the
//               other roles through a 2-entry shared-memory ring, and loads
//               each item's Q_A/Q_B once the previous item's last S is done
//   warps 12-15 epilogue: when a side has reported an item's last P, it hands
//               each row's sum l and reference maximum m to these warps
//               through a shared-memory slot and goes straight on to the next
//               item; they wait for the side's last product, read O out of
//               TMEM, release it to the next item's products, normalise,
//               pack and store each row
// The producers' lanes resolve a tile's blocks through the block table and
// issue one TMA box each (blocks of fewer than 8 rows: 16-byte cp.async).
// Registers (setmaxnreg, each warpgroup at the top of its own branch): the
// softmax warpgroups 200 each, the producer/MMA/scheduler warpgroup 64 and
// the epilogue warpgroup 48, which adds up to the 4 x 128 a thread is
// launched with (per SM sub-partition 200+200+64+48 registers x 32 lanes =
// 16384).  A launch of 512 threads compiles every single instruction within
// 128 registers, so a softmax row of 128 scores is read from TMEM as two
// 64-column loads; the MMA lane keeps each shared-memory descriptor as one
// 32-bit word to fit in its 64.
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512).
// P (bf16, two per 32-bit column) is written over the first 64 columns of its
// own S and read from there as the A operand of O += P V.  Per key tile j the
// tensor core runs, in issue order, PV_A(j) S_A(j+1) PV_B(j) S_B(j+1), so while
// softmax A works on S_A(j+1) it computes B's products and the other way round
// (the two tiles ping-pong).  tcgen05.mma operations issued by one thread run
// in order, so S(j+1) overwrites P(j) only after PV(j) has read it, and the
// commit that reports S(j+1) also reports every earlier product: a softmax
// thread that has S(j+1) may rewrite its P columns and rescale its O.
// S = Q K^T reads both operands from 128-byte-swizzled shared memory; V is read
// MN-major.

// Online softmax: the running max m of a row only moves when the tile maximum
// exceeds it by more than 8 (a factor 256 in base 2); O and l are then scaled
// by 2^(m_old - m_new).  Numerator and denominator use the same m, so the
// result is exact for any m; the threshold only bounds P <= 256.  Scores are in
// the log2 domain (scale pre-multiplied by log2 e).
//
// Every mbarrier wait is bounded (2 s, or the limit pa_set_wait_limit_ns
// set); on expiry the kernel sets PA_DEV_TIMEOUT, drains its in-flight copies
// and MMAs (each drain wait bounded at 2 s), frees TMEM and exits.
#include <cuda.h>
#include <limits.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace pa {

namespace {

using namespace tc;

constexpr int kM = 128;  // query rows per tile (TMEM lanes)
constexpr int kN = 128;  // keys per tile
constexpr int kSoftmaxWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kVWarp = 10;
constexpr int kSchedWarp = 11;
constexpr int kEpiWarp0 = 12;  // warps 12-15: epilogue
constexpr int kThreads = 512;
// setmaxnreg split of the 128 registers a thread is launched with
constexpr int kSoftmaxRegs = 200;
constexpr int kProducerRegs = 64;
constexpr int kEpiRegs = 48;
static_assert(2 * kSoftmaxRegs + kProducerRegs + kEpiRegs == 4 * 65536 / kThreads,
              "the warpgroups' register limits must add up to the launch's");
// With the fused scatter the producers carry more state: 8 more registers
// for them, 8 fewer for the epilogue.
constexpr int kProducerRegsFused = 72;
constexpr int kEpiRegsFused = 40;
static_assert(2 * kSoftmaxRegs + kProducerRegsFused + kEpiRegsFused == 4 * 65536 / kThreads,
              "the warpgroups' register limits must add up to the launch's");
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitNs = 2000000000ull;

// ---- fp32 pairs ------------------------------------------------------------------
// The softmax works on pairs of scores with the f32x2 add / fma instructions
// of this architecture, and takes row maxima three operands at a time; both
// cut its instruction count, which (not the exponential unit) bounds it.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};\n" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_split(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;\n" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// The scheduler's table of items per cost level (ints, in shared memory);
// with more levels it scans the slots instead.
constexpr int kMaxLevels = 2048;

template <int D>
struct PpLayout {
  static constexpr int kHalves = D / 64;        // 64-element (128-byte) column chunks
  static constexpr int kHalf = kM * 128;         // one chunk of a 128-row tile: 16 KB
  static constexpr int kTile = kHalves * kHalf;  // Q, K or V tile
  static constexpr int kKStages = 2;
  static constexpr int kVStages = 2;
  static constexpr int kQ = 0;  // Q of side A, then of side B
  static constexpr int kK = 2 * kTile;
  static constexpr int kV = kK + kKStages * kTile;
  static constexpr int kEpi = kV + kVStages * kTile;  // softmax -> epilogue hand-off slots
  static constexpr int kBar = kEpi + 5 * 1024;
  static constexpr int kLv = kBar + 512;  // after the barriers, TMEM slot, flags, item ring
  static constexpr int kBytes = kLv + 4 * kMaxLevels;  // the scheduler's level table
  static constexpr int kAlloc = kBytes + 1024;   // slack to align the base to 1 KB
  static_assert(kAlloc <= 227 * 1024, "shared memory per CTA");
  __host__ __device__ static constexpr int q(int side) { return kQ + side * kTile; }
};

enum : int {
  bQFull, bQFree,
  bKFull0, bKFull1, bKEmpty0, bKEmpty1,
  bVFull0, bVFull1, bVEmpty0, bVEmpty1,
  bSA, bSB, bPA, bPB, bPvA, bPvB, bOFreeA, bOFreeB, bDrain,
  bItemFull0, bItemFull1, bItemEmpty0, bItemEmpty1, bLA0, bLA1, bLB0, bLB1, kNumBars
};


// Arrivals that release each item's ring entry: one lane of the K producer,
// the MMA and the V producer warps, and every softmax thread.
constexpr uint32_t kItemReaders = 3 + 32 * kSoftmaxWarps;
// The barrier area: the mbarriers, then the TMEM address, the abort flag and
// the epilogue's stop word (4 bytes each), then the 2-entry item ring.
constexpr int kRingOffset = (8 * kNumBars + 12 + 15) / 16 * 16;

struct Item {
  int s, hk, h[2], t0, qn, c, i0, kv_end, n;  // h[1] < 0: no second tile
  int nh;  // fused scatter: tiles of cached history before the new-token tiles (else 0)
  int pk;  // packed: a tile of <= 64 query tokens holds two heads (rows 0-63: head
           // h, rows 64-127: head h + 1), so the item covers four heads
};

static_assert(kRingOffset + 2 * static_cast<int>(sizeof(Item)) <= 512,
              "barriers, flags and item ring must fit the 512-byte barrier area");

// What a softmax side hands to the epilogue warps when it has reported an
// item's last P: each row's sum l and reference maximum m (log2 domain), and
// the item (n = 0 in side A's slot: no more items).  Two slots per side, by
// the side's item parity.
struct EpiSlot {
  float l[kM];
  float m[kM];
  Item it;
};
static_assert(4 * sizeof(EpiSlot) <= 5 * 1024, "hand-off slots");

// Key range [key0, key_end) of tile j of an item.  Without the fused scatter
// the tiles are 128-position windows from position 0.  With it, the cached
// history c comes first in 128-position windows (the last one cut at c),
// then the new tokens in 128-position windows starting at c, so that every
// new-token tile is 128 consecutive input rows.
__device__ __forceinline__ void tile_keys(const Item& I, int j, bool fused, int& key0,
                                          int& key_end, bool casc = false) {
  if (casc) {  // a chunk [c, kv_end) of a shared prefix
    key0 = I.c + j * kN;
    key_end = min(key0 + kN, I.kv_end);
  } else if (fused && j >= I.nh) {
    key0 = I.c + (j - I.nh) * kN;
    key_end = min(key0 + kN, I.kv_end);
  } else {
    key0 = j * kN;
    key_end = min(key0 + kN, fused ? I.c : I.kv_end);
  }
}

// Next count from a (tag << 32 | count) word of the work queue.  A word that
// holds another launch's tag, or a count no draw of this launch can reach
// (bound), is reset by the first CTA that manages to: it reads the word and
// swaps exactly what it read for (tag, 1), taking 0.  A CTA adds to a stale
// word at most once (its first try, which is the common case's only atomic),
// so the swaps cannot be kept failing by other CTAs' additions for long.
// False after many lost swaps (the caller reports it).
__device__ bool tagged_take(unsigned long long* w, uint32_t tag, uint32_t bound, uint32_t& n) {
  const unsigned long long mine = static_cast<unsigned long long>(tag) << 32;
  auto fresh = [&](unsigned long long v) {
    return (v >> 32) == tag && static_cast<uint32_t>(v) < bound;
  };
  unsigned long long v = atomicAdd(w, 1ull);
  for (int tries = 0; tries < 4096; ++tries) {
    if (fresh(v)) {
      n = static_cast<uint32_t>(v);
      return true;
    }
    const unsigned long long cur = atomicOr(w, 0ull);  // read
    if (fresh(cur)) {
      v = atomicAdd(w, 1ull);
    } else if (atomicCAS(w, cur, mine | 1ull) == cur) {
      n = 0;
      return true;
    }
  }
  return false;
}

// Query tokens [t0, t0 + qn) and length L of sequence s; false when it has
// no query tokens or its metadata is out of range (bad).
__device__ __forceinline__ bool seq_rows(const AttnArgs& a, int s, int& t0, int& qn, int& L,
                                         bool& bad) {
  t0 = __ldg(a.qsl + s);
  qn = __ldg(a.qsl + s + 1) - t0;
  L = __ldg(a.seq_lens + s);
  bad = false;
  if (qn <= 0) return false;
  if (L < qn || L > (a.max_blocks << a.bs_log2) || qn > a.max_query_len || L > a.max_seq_len ||
      t0 < 0 || t0 + qn > a.num_tokens) {
    bad = true;
    return false;
  }
  return true;
}

// Cost levels of prefill sequence sp's token tiles: tile t has level lo + t
// (t < nt); pk_last: the last tile is packed (at most 64 tokens, group of
// four heads).  Every level is at most ceil(max_seq_len / 128) + 1.
__device__ __forceinline__ bool seq_levels(const AttnArgs& a, int sp, int& lo, int& nt,
                                           bool& pk_last, bool& bad) {
  int t0, qn, L;
  if (!seq_rows(a, a.num_decode + sp, t0, qn, L, bad)) return false;
  lo = (L - qn + kN - 1) / kN + 1;
  nt = (qn + kM - 1) / kM;
  pk_last = qn - (nt - 1) * kM <= kM / 2 && a.group % 4 == 0;
  return true;
}

// Work slot e -> item.  Slots enumerate (cost level from max_level down to 1,
// sequence, kv head, head pair); the sequence's tile at that level is
// t = level - 1 - ceil(c / 128); a slot whose tile does not exist is empty.
template <bool kFused>
__device__ bool decode_item(const AttnArgs& a, int e, int pairs, int max_level, Item& it,
                            bool& bad) {
  const int S_pre = a.num_seqs - a.num_decode;
  const int per_seq = a.hkv * pairs;
  const int per_z = per_seq * S_pre;
  const int z = e / per_z;
  int rest = e - z * per_z;
  const int sp = rest / per_seq;
  rest -= sp * per_seq;
  const int hk = rest / pairs;
  const int p = rest - hk * pairs;
  const int s = a.num_decode + sp;
  int t0, qn, L;
  if (!seq_rows(a, s, t0, qn, L, bad)) return false;
  const int level = max_level - z;
  const int tile = level - 1 - (L - qn + kN - 1) / kN;
  if (tile < 0 || tile >= (qn + kM - 1) / kM) return false;
  // A tile of at most 64 tokens takes two heads per side (when the group
  // splits into fours): half the products for the same rows.
  const bool pk = qn - tile * kM <= kM / 2 && a.group % 4 == 0;
  if (pk && 4 * p >= a.group) return false;
  it.s = s;
  it.hk = hk;
  it.pk = pk ? 1 : 0;
  if (pk) {
    it.h[0] = hk * a.group + 4 * p;
    it.h[1] = it.h[0] + 2;
  } else {
    it.h[0] = hk * a.group + 2 * p;
    it.h[1] = 2 * p + 1 < a.group ? it.h[0] + 1 : -1;
  }
  it.t0 = t0;
  it.qn = qn;
  it.c = L - qn;
  it.i0 = tile * kM;
  it.kv_end = it.c + min(qn, it.i0 + kM);
  if (kFused) {
    it.nh = (it.c + kN - 1) / kN;
    it.n = it.nh + it.i0 / kN + 1;
  } else {
    it.nh = 0;
    it.n = (it.kv_end + kN - 1) / kN;
  }
  return true;
}

// Shared-prefix (cascade) prefix pass: slot e -> (kv head, pair of 128-row
// query tiles, key chunk of the prefix).  Query row r of kv head hk is
// (decode sequence r / g, query head hk * g + r % g).  Fields: h = the two
// tiles (h[1] < 0: none), c / kv_end = the chunk's keys, t0 = the chunk's
// partial slot, qn = the kv head's row count, s = 0 (the prefix blocks are
// read through the first sequence's table).
__device__ bool decode_item_casc(const AttnArgs& a, int e, Item& it) {
  const int rows = a.num_decode * a.group;
  const int tiles = (rows + kM - 1) / kM;
  const int tpairs = (tiles + 1) / 2;
  const int per_hk = tpairs * a.nsplit_prefix;
  const int hk = e / per_hk;
  const int rest = e - hk * per_hk;
  const int tp = rest / a.nsplit_prefix;
  const int ch = rest - tp * a.nsplit_prefix;
  const int k_lo = ch * a.part_prefix;
  const int k_hi = min(a.prefix_len, k_lo + a.part_prefix);
  if (hk >= a.hkv || k_lo >= k_hi) return false;
  it.s = 0;
  it.hk = hk;
  it.h[0] = 2 * tp;
  it.h[1] = 2 * tp + 1 < tiles ? 2 * tp + 1 : -1;
  it.t0 = ch;
  it.qn = rows;
  it.c = k_lo;
  it.i0 = 0;
  it.kv_end = k_hi;
  it.nh = 0;
  it.pk = 0;
  it.n = (k_hi - k_lo + kN - 1) / kN;
  return true;
}

// kPoll: the instantiation launched when an explicit wait limit is set
// (pa_set_wait_limit_ns): every wait polls without suspending, so that even a
// limit of a few nanoseconds holds.  The default instantiation's first probe
// of a barrier may suspend inside the hardware until the phase completes.
template <int D, bool kFused, bool kCasc = false, bool kPoll = false>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_o,
                      const __grid_constant__ CUtensorMap tm_kn,
                      const __grid_constant__ CUtensorMap tm_vn,
                      const __grid_constant__ CUtensorMap tm_q64, const AttnArgs a,
                      int total_slots, int max_level) {
  using Ly = PpLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pairs = (a.group + 1) >> 1;

  const uint32_t bar0 = base + Ly::kBar;
  const uint32_t tmem_slot = bar0 + 8 * kNumBars;
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(sgen + Ly::kBar + 8 * kNumBars + 4);
  // items side A has handed to the epilogue warps when it runs out of items
  volatile int* epi_total = reinterpret_cast<volatile int*>(sgen + Ly::kBar + 8 * kNumBars + 8);
  Item* ring = reinterpret_cast<Item*>(sgen + Ly::kBar + kRingOffset);
#define BAR(i) (bar0 + 8u * static_cast<uint32_t>(i))

  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      const bool many = i == bPA || i == bPB || i == bOFreeA || i == bOFreeB || i == bLA0 ||
                        i == bLA1 || i == bLB0 || i == bLB1;
      const bool readers = i == bItemEmpty0 || i == bItemEmpty1;
      mbar_init(BAR(i), many ? 128u : (readers ? kItemReaders : 1u));
    }
    *abort_flag = 0u;
    *epi_total = INT_MAX;
    fence_barrier_init();
  }
  if (!kCasc && warp == kSchedWarp && lane < a.num_seqs - a.num_decode) {
    // the scheduler's first reads: the first prefill sequences' metadata
    prefetch_l1(a.qsl + a.num_decode + lane);
    prefetch_l1(a.qsl + a.num_decode + lane + 1);
    prefetch_l1(a.seq_lens + a.num_decode + lane);
  }
  if (threadIdx.x == 32 * kProducerWarp) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_o);
    if (kFused) {
      prefetch_tmap(&tm_kn);
      prefetch_tmap(&tm_vn);
    }
    if (!kCasc) prefetch_tmap(&tm_q64);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sgen + Ly::kBar + 8 * kNumBars);

  auto give_up = [&]() {
    *abort_flag = 1u;
    flag_error(a.err, PA_DEV_TIMEOUT);
  };
  auto wait = [&](int b, int completion) -> bool {
    const uint32_t parity = static_cast<uint32_t>(completion) & 1u;
    if constexpr (kPoll) {
      if (mbar_test_wait(BAR(b), parity)) return true;
    } else {
      if (mbar_try_wait(BAR(b), parity)) return true;
    }
    if (*abort_flag) return false;
    if (mbar_wait(BAR(b), parity, a.wait_ns ? a.wait_ns : kWaitNs)) return true;
    give_up();
    return false;
  };

  // Waits of the warp-collective roles (softmax, producers).  Under a short
  // explicit limit (kPoll) one lane's wait can run out while another's sees
  // the phase complete; the warp then takes the outcome together, so that no
  // lane is left alone at a warp-wide instruction (tcgen05.ld/st, shuffles,
  // __syncwarp).  Under the default 2 s limit every lane polls the same phase,
  // so the lanes give up together unless it completes within the same
  // microsecond; the waits stay per lane there, without a vote.
  auto wait_w = [&](int b, int completion) -> bool {
    if constexpr (kPoll) return __all_sync(0xffffffffu, wait(b, completion));
    else return wait(b, completion);
  };

  // Take item number `it` from the ring (every lane of a reading warp calls
  // this); `arrive`: this thread reports the entry consumed.
  auto next_item = [&](int it, Item& I, bool arrive) -> bool {
    const int slot = it & 1;
    if (!wait_w(bItemFull0 + slot, it >> 1)) return false;
    I = ring[slot];  // ordered after the acquiring wait (asm with a memory clobber)
    if (arrive) mbar_arrive(BAR(bItemEmpty0 + slot));
    return I.n > 0;
  };

  // The Q boxes of an item.  A packed item has two heads per side in 64-row
  // boxes (tm_q64).
  auto q_copy = [&](const Item& I) {
    const uint32_t full = BAR(bQFull);
    if (I.pk) {
#pragma unroll
      for (int hf = 0; hf < Ly::kHalves; ++hf)
#pragma unroll
        for (int u = 0; u < 4; ++u)  // heads h[0], h[0]+1 (side A), h[1], h[1]+1 (side B)
          tma_load_2d(base + Ly::q(u >> 1) + hf * Ly::kHalf + (u & 1) * (kM / 2) * 128,
                      &tm_q64, (I.h[u >> 1] + (u & 1)) * D + hf * 64, I.t0 + I.i0, full);
    } else {
#pragma unroll
      for (int hf = 0; hf < Ly::kHalves; ++hf)
#pragma unroll
        for (int sd = 0; sd < 2; ++sd)
          if (sd == 0 || I.h[1] >= 0)
            tma_load_2d(base + Ly::q(sd) + hf * Ly::kHalf, &tm_q, I.h[sd] * D + hf * 64,
                        I.t0 + I.i0, full);
    }
  };

  EpiSlot* epi = reinterpret_cast<EpiSlot*>(sgen + Ly::kEpi);  // [parity][side]
  // Each warpgroup's register limit is set at the top of its own branch, so
  // that the compiler allocates each role's code within its own limit.
  if (warp >= kProducerWarp && warp < kEpiWarp0) {
  regs_decrease<kFused ? kProducerRegsFused : kProducerRegs>();
  if (warp == kSchedWarp) {
    // ------------------------------------------------------------ scheduler
    // Dense work list: the global counter numbers only the items that exist,
    // in slot order (cost level from the top, sequence, kv head, head pair),
    // so every draw yields an item.  The warp first tabulates, per level z,
    // lv[z] = the number of items at levels <= z (a difference array over
    // each sequence's level range, summed twice); draw d then lies at level
    // z, the smallest with lv[z] >= total - d, and is the (lv[z] - total + d)-th
    // item of that level, found by a scan over the sequences.  With too many
    // levels for the table, the counter walks the slots and skips empty ones.
    constexpr unsigned kAll = 0xffffffffu;
    int* lv = reinterpret_cast<int*>(sgen + Ly::kLv);
    const int S_pre = a.num_seqs - a.num_decode;
    const int M = a.hkv * pairs;            // items of one sequence at one level
    const int Mp = a.hkv * (a.group >> 2);  // the same, packed tile
    const bool dense = !kCasc && max_level + 2 <= kMaxLevels;
    // The work counter as this launch finds it; read now, used after the
    // table is built (see below).
    unsigned long long seen = 0;
    if (lane == 0) seen = atomicOr(a.sched, 0ull);
    int total_items = 0;
    if (dense) {
      for (int z = lane; z < max_level + 2; z += 32) lv[z] = 0;
      __syncwarp();
      for (int sp = lane; sp < S_pre; sp += 32) {
        int lo, nt;
        bool pkl, bad;
        if (seq_levels(a, sp, lo, nt, pkl, bad)) {
          atomicAdd(lv + lo, M);
          atomicAdd(lv + lo + nt, -M);
          if (pkl) {
            atomicAdd(lv + lo + nt - 1, Mp - M);
            atomicAdd(lv + lo + nt, M - Mp);
          }
        } else if (bad) {
          flag_error(a.err, PA_DEV_BAD_LEN);
        }
      }
      __syncwarp();
      int run1 = 0, run2 = 0;  // items at the levels so far; their running sum
      for (int z0 = 0; z0 <= max_level; z0 += 32) {
        const int z = z0 + lane;
        int v = z <= max_level ? lv[z] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(kAll, v, o);
          if (lane >= o) v += u;
        }
        int w = run1 + v;  // items at level z
        run1 += __shfl_sync(kAll, v, 31);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(kAll, w, o);
          if (lane >= o) w += u;
        }
        if (z <= max_level) lv[z] = run2 + w;
        run2 += __shfl_sync(kAll, w, 31);
      }
      __syncwarp();
      total_items = lv[max_level];
    }
    // Slot of the d-th item of the dense list (every lane; -1: not found,
    // which only metadata changing under the kernel could cause).
    auto dense_slot = [&](int d) -> int {
      const int u = total_items - d;
      int zl = 1, zh = max_level;
      while (zl < zh) {
        const int mid = (zl + zh) >> 1;
        if (lv[mid] >= u) zh = mid;
        else zl = mid + 1;
      }
      const int z = zl;
      const int k = lv[z] - u;
      int acc = 0;
      for (int s0 = 0; s0 < S_pre; s0 += 32) {
        const int sp = s0 + lane;
        int m = 0;
        bool pk = false;
        if (sp < S_pre) {
          int lo, nt;
          bool pkl, bad;
          if (seq_levels(a, sp, lo, nt, pkl, bad) && z >= lo && z < lo + nt) {
            pk = pkl && z == lo + nt - 1;
            m = pk ? Mp : M;
          }
        }
        int incl = m;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u2 = __shfl_up_sync(kAll, incl, o);
          if (lane >= o) incl += u2;
        }
        const int tot = __shfl_sync(kAll, incl, 31);
        if (k < acc + tot) {
          const int src = __ffs(__ballot_sync(kAll, k < acc + incl)) - 1;
          const int r = k - acc - __shfl_sync(kAll, incl - m, src);
          const int mult = __shfl_sync(kAll, static_cast<int>(pk), src) ? (a.group >> 2) : pairs;
          return ((max_level - z) * S_pre + s0 + src) * M + (r / mult) * pairs + r % mult;
        }
        acc += tot;
      }
      return -1;
    };
    // The next item of this CTA (every lane; I.n = 0: none left).  The first
    // draw of CTA b is number b; the work counter numbers the draws after the
    // first wave.  Every CTA with a first item draws until a draw comes back
    // past the list (T numbers: items, or slots), so a launch makes exactly T
    // counted draws whatever the timing, and the CTA that draws count T - 1
    // made the last one: it leaves the word at (tag, 0), so that a replay of
    // the same launch (a CUDA graph keeps its arguments) starts from 0.
    bool first = true;
    const uint32_t T = static_cast<uint32_t>(dense ? total_items : total_slots);
    // A counter left by another launch is reset before the first wave
    // draws from it: each CTA swaps exactly the stale value it read for
    // (tag, 0), so only the first swap takes effect and none can undo a draw.
    // A CTA that draws before any swap has landed resets it in tagged_take.
    if (lane == 0 && !((seen >> 32) == a.sched_tag && static_cast<uint32_t>(seen) < T))
      atomicCAS(a.sched, seen, static_cast<unsigned long long>(a.sched_tag) << 32);
    auto draw = [&](Item& I) {
      I.n = 0;
      while (true) {
        unsigned e0 = 0;
        if (first) {
          e0 = blockIdx.x;
        } else if (lane == 0) {
          uint32_t n;
          if (tagged_take(a.sched, a.sched_tag, T, n)) {
            e0 = gridDim.x + n;
            if (n == T - 1) atomicExch(a.sched, static_cast<unsigned long long>(a.sched_tag) << 32);
          } else {
            flag_error(a.err, PA_DEV_TIMEOUT);
            e0 = 0x7fffffffu;  // no more items for this CTA
          }
        }
        first = false;
        const int e = static_cast<int>(__shfl_sync(kAll, e0, 0));
        bool bad = false;
        if constexpr (kCasc) {
          if (e >= total_slots) return;
          if (decode_item_casc(a, e, I)) return;
        } else if (dense) {
          if (e >= total_items) return;
          const int slot = dense_slot(e);
          if (slot >= 0 && decode_item<kFused>(a, slot, pairs, max_level, I, bad)) return;
        } else {
          if (e >= total_slots) return;
          if (decode_item<kFused>(a, e, pairs, max_level, I, bad)) return;
          if (bad && lane == 0) flag_error(a.err, PA_DEV_BAD_LEN);
        }
      }
    };
    int q_issued = 0;
    bool drawn_out = false;  // a draw came back past the list
    for (int it = 0;; ++it) {
      Item I;
      draw(I);
      drawn_out = I.n <= 0;
      int stop = 0;
      if (lane == 0) {
        const int slot = it & 1;
        if (it >= 2 && !wait(bItemEmpty0 + slot, (it >> 1) - 1)) {
          stop = 1;
        } else {
          ring[slot] = I;  // published by the releasing arrive below
          mbar_arrive(BAR(bItemFull0 + slot));  // release: the entry is visible to waiters
          // Q of this item, into the Q buffers the previous item has finished with
          if (I.n <= 0 || (it > 0 && !wait(bQFree, it - 1))) stop = 1;
        }
        if (!stop) {
          const bool hasB = I.h[1] >= 0;
          mbar_expect_tx(BAR(bQFull), Ly::kTile * (hasB ? 2 : 1));
          if constexpr (kCasc) {
            // a tile's rows come g at a time: the g query heads of kv head hk
            // of one decode token (tm_q is [tokens, heads, D] here, box g heads);
            // rows past the last sequence read an out-of-range token (zeros)
            for (int sd = 0; sd < (hasB ? 2 : 1); ++sd) {
              const uint32_t qdst = base + Ly::q(sd);
              for (int rb = 0; rb < kM; rb += a.group) {
                const int seq = (I.h[sd] * kM + rb) / a.group;
                int t0 = seq < a.num_decode ? __ldg(a.qsl + seq) : a.num_tokens;
                if (t0 < 0 || t0 >= a.num_tokens) t0 = a.num_tokens;
#pragma unroll
                for (int hf = 0; hf < Ly::kHalves; ++hf)
                  tma_load_3d(qdst + hf * Ly::kHalf + rb * 128, &tm_q, hf * 64, I.hk * a.group,
                              t0, BAR(bQFull));
              }
            }
          } else {
            q_copy(I);
          }
          q_issued = it + 1;
        }
      }
      if (__shfl_sync(kAll, stop, 0)) break;
    }
    // A CTA that gave up mid-way still draws to the end of the list (without
    // running the items), which keeps the count of draws at T.
    while (!drawn_out) {
      Item I;
      draw(I);
      drawn_out = I.n <= 0;
    }
    // drain: the last Q copy has landed before the CTA exits (each earlier
    // one was consumed before the next was issued)
    if (lane == 0 && q_issued > 0) mbar_wait(BAR(bQFull), (q_issued - 1) & 1, kWaitNs);
    __syncwarp();
  } else if (warp == kProducerWarp || warp == kVWarp) {
    // ------------------------------------------------------------ producers
    // warp 8: the K tiles; warp 10: the V tiles.  Cached positions come from
    // the paged cache, one TMA box per block (lane b issues box b).  With the
    // fused scatter, the new tokens' tiles (see tile_keys) are 128
    // consecutive rows of the new-token K/V: one box per 64-column half.
    // Items of the first head pair then store their own query rows' K (V)
    // into their slots, read back from the item's last tile in shared memory.
    const bool is_k = warp == kProducerWarp;
    const int nst = is_k ? Ly::kKStages : Ly::kVStages;
    const int full0 = is_k ? bKFull0 : bVFull0;
    const int empty0 = is_k ? bKEmpty0 : bVEmpty0;
    const uint32_t stage0 = base + (is_k ? Ly::kK : Ly::kV);
    const CUtensorMap* map = is_k ? &tm_k : &tm_v;
    const CUtensorMap* nmap = is_k ? &tm_kn : &tm_vn;
    constexpr bool fused = kFused;
    constexpr int kCpr = D / 8;  // 16-byte pieces per row
    int gt = 0, it = 0, last = -1;
    // Pending store of an item's own rows (fused scatter): the tile holding
    // them and the item.  Lane r stores rows r, r + 32, ... (one slot each,
    // 16-byte pieces in order), which keeps the instruction count low: this
    // warp shares its sub-partition with two softmax warps.  The store runs
    // while this warp would otherwise wait for a free stage, and at the
    // latest before that tile's stage is refilled.
    int pend_g = -1;
    int pend_row0 = 0, pend_rows = 0, pend_hk = 0;  // first input row, row count, kv head
    auto scatter = [&]() -> bool {
      const int g = pend_g;
      if (!wait_w(full0 + g % nst, g / nst)) return false;
      const uint8_t* sg = sgen + (stage0 - base) + (g % nst) * Ly::kTile;
      const int64_t nslots = static_cast<int64_t>(a.num_blocks) << a.bs_log2;
      __nv_bfloat16* cw = static_cast<__nv_bfloat16*>(const_cast<void*>(is_k ? a.k_cache : a.v_cache)) +
                          static_cast<int64_t>(pend_hk) * D;
#pragma unroll 1
      for (int r = lane; r < pend_rows; r += 32) {
        const int sl = __ldg(a.slots + pend_row0 + r);
        if (sl >= nslots) {
          flag_error(a.err, PA_DEV_BAD_SLOT);
        } else if (sl >= 0) {
          uint4* dst = reinterpret_cast<uint4*>(cw + static_cast<int64_t>(sl) * a.hkv * D);
          const uint8_t* src = sg + r * 128;
#pragma unroll
          for (int c16 = 0; c16 < kCpr; ++c16)
            dst[c16] = *reinterpret_cast<const uint4*>(src + (c16 >> 3) * Ly::kHalf +
                                                        (((c16 & 7) ^ (r & 7)) << 4));
        }
      }
      __syncwarp();
      pend_g = -1;
      return true;
    };
    // Before waiting for stage st of tile gt.
    auto before_refill = [&](int st) -> bool {
      if (pend_g < 0) return true;
      if (st != pend_g % nst) {  // optional: only while the stage is busy and the rows are in
        const bool busy = gt >= nst && !__all_sync(0xffffffffu, mbar_test_wait(BAR(empty0 + st),
                                                                              (gt / nst - 1) & 1));
        const bool landed = __all_sync(0xffffffffu, mbar_test_wait(BAR(full0 + pend_g % nst),
                                                                  (pend_g / nst) & 1));
        if (!busy || !landed) return true;
      }
      return scatter();
    };
    const int bs = 1 << a.bs_log2;
    const int R = bs < kN ? bs : kN;  // cache rows per TMA box; lane b owns box b
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Item I;
      if (!next_item(k, I, false)) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(bItemEmpty0 + (k & 1)));
      ++it;
      const int32_t* bt = a.block_tables + static_cast<int64_t>(I.s) * a.max_blocks;
      const int64_t head = static_cast<int64_t>(I.hk) * D;
      for (int j = 0; j < I.n; ++j, ++gt) {
        const int st = gt % nst;
        int key0, key_end;
        tile_keys(I, j, fused, key0, key_end, kCasc);
        const uint32_t stile = stage0 + st * Ly::kTile;
        if (fused && j >= I.nh) {
          // new tokens: input rows t0 + (key0 - c) ..., one 128-row box per half
          if (!(ok = before_refill(st))) break;
          if (gt >= nst && !(ok = wait_w(empty0 + st, gt / nst - 1))) break;
          if (lane == 0) {
            mbar_expect_tx(BAR(full0 + st), kN * 128 * Ly::kHalves);
#pragma unroll
            for (int hf = 0; hf < Ly::kHalves; ++hf)
              tma_load_2d(stile + hf * Ly::kHalf, nmap, static_cast<int>(head) + hf * 64,
                          I.t0 + (key0 - I.c), BAR(full0 + st));
          }
          __syncwarp();
          last = gt;
          continue;
        }
        if (bs < 8) {
          // Blocks of fewer than 8 rows: a box would not fill whole 8-row
          // swizzle atoms, so the lanes gather the rows themselves with
          // 16-byte cp.async into the same 128-byte-swizzled layout (lane l
          // takes rows l, l + 32, ...), wait for their own copies and make
          // them visible to the tensor core (proxy fence) before lane 0
          // reports the stage full.  Rows past the tile's last key are left
          // as they are, as with boxes.
          if (!(ok = before_refill(st))) break;
          if (gt >= nst && !(ok = wait_w(empty0 + st, gt / nst - 1))) break;
          const char* cbase = static_cast<const char*>(is_k ? a.k_cache : a.v_cache);
#pragma unroll 1
          for (int rr = lane; rr < key_end - key0; rr += 32) {
            const int pos = key0 + rr;
            const int pb = __ldg(bt + (pos >> a.bs_log2));
            if (pb < 0 || pb >= a.num_blocks) {
              flag_error(a.err, PA_DEV_BAD_BLOCK);
              continue;
            }
            const int64_t sl = (static_cast<int64_t>(pb) << a.bs_log2) + (pos & (bs - 1));
            const char* src = cbase + (sl * a.hkv + I.hk) * (D * 2);
            const uint32_t drow = stile + rr * 128;
#pragma unroll
            for (int c = 0; c < kCpr; ++c)
              cp_async16(drow + (c >> 3) * Ly::kHalf + (((c & 7) ^ (rr & 7)) << 4), src + c * 16,
                         true);
          }
          cp_async_commit();
          cp_async_wait<0>();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(full0 + st));
          last = gt;
          continue;
        }
        // cached positions: one box per block
        const int nbox = (key_end - key0 + R - 1) / R;
        int slot = -1;
        const int b = lane;
        if (b < nbox) {
          const int pos = key0 + b * R;
          const int pb = __ldg(bt + (pos >> a.bs_log2));
          if (pb >= 0 && pb < a.num_blocks) slot = (pb << a.bs_log2) + (pos & (bs - 1));
          else flag_error(a.err, PA_DEV_BAD_BLOCK);
        }
        const uint32_t valid = __ballot_sync(0xffffffffu, slot >= 0);
        const uint32_t bytes = static_cast<uint32_t>(__popc(valid) * R * 128 * Ly::kHalves);
        if (!(ok = before_refill(st))) break;
        if (gt >= nst && !(ok = wait_w(empty0 + st, gt / nst - 1))) break;
        if (lane == 0) mbar_expect_tx(BAR(full0 + st), bytes);
        __syncwarp();
        if (slot >= 0) {
          const uint32_t dst = stile + b * R * 128;
#pragma unroll
          for (int hf = 0; hf < Ly::kHalves; ++hf)
            tma_load_3d(dst + hf * Ly::kHalf, map, hf * 64, I.hk, slot, BAR(full0 + st));
        }
        last = gt;
      }
      if (!ok) break;
      if (fused && I.h[0] == I.hk * a.group) {
        // The item's last tile holds its own query rows' K (V) as rows
        // 0 .. rows - 1: store them into their slots once it has landed.
        if (pend_g >= 0 && !(ok = scatter())) break;
        pend_g = gt - 1;
        pend_row0 = I.t0 + I.i0;
        pend_rows = min(kM, I.qn - I.i0);
        pend_hk = I.hk;
      }
    }
    if (ok && pend_g >= 0) ok = scatter();
    // drain: every copy this warp issued has landed before the CTA exits
    if (lane == 0) {
      for (int t = max(0, last - nst + 1); t <= last; ++t)
        mbar_wait(BAR(full0 + t % nst), (t / nst) & 1, kWaitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_bf16(kM, kN, false);
    constexpr uint32_t kIdO = idesc_bf16(kM, D, true);
    // Shared-memory descriptors are built once; a K step or a stage moves the
    // start address, which sits in the descriptor's low bits (address >> 4),
    // so each product costs one add per operand.  (The issuing lane shares its
    // sub-partition with two softmax warps, so every instruction it saves
    // shortens the gap between a P being ready and its product starting.)
    const uint64_t dQ0 = smem_desc_sw128(base + Ly::kQ, 16, 1024);
    const uint64_t dK0 = smem_desc_sw128(base + Ly::kK, 16, 1024);
    const uint64_t dV0 = smem_desc_sw128(base + Ly::kV, Ly::kHalf, 1024);
    const uint32_t dHi = static_cast<uint32_t>(dQ0 >> 32);  // the same for all three
    const uint32_t tS0 = tmem, tO0 = tmem + 256;
    // S of one side for key tile g
    auto issue_s = [&](int side, int g) {
      const uint32_t a0 = opaque_u32(static_cast<uint32_t>(dQ0) + (Ly::q(side) >> 4));
      const uint32_t b0 = opaque_u32(static_cast<uint32_t>(dK0) +
                                     (g % Ly::kKStages) * (Ly::kTile >> 4));
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * Ly::kHalf + (kk & 3) * 32) >> 4;
        mma_f16_ss_lo(tS0 + side * 128, a0 + off, b0 + off, dHi, kIdS, kk > 0 ? 1u : 0u);
      }
      mma_commit(BAR(side ? bSB : bSA));
    };
    auto issue_pv = [&](int side, int g, bool acc) {
      const uint32_t v0 = opaque_u32(static_cast<uint32_t>(dV0) +
                                     (g % Ly::kVStages) * (Ly::kTile >> 4));
#pragma unroll
      for (int kk = 0; kk < kN / 16; ++kk)
        mma_f16_ts_lo(tO0 + side * 128, tS0 + side * 128 + kk * 8, v0 + kk * (2048 >> 4), dHi,
                      kIdO, (acc || kk > 0) ? 1u : 0u);
    };
    // One lane issues everything; the V rows past the last key of a partial
    // tile are zeroed by softmax A before it reports its P.  This lane needs
    // only an item's tile count and whether it has a side B.
    auto next_nb = [&](int it, int& n, bool& hb) -> bool {
      const int slot = it & 1;
      if (!wait(bItemFull0 + slot, it >> 1)) return false;
      n = ring[slot].n;
      hb = ring[slot].h[1] >= 0;
      mbar_arrive(BAR(bItemEmpty0 + slot));
      return n > 0;
    };
    if (lane == 0) {
      int gt = 0, it = 0, gB = 0, itB = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        int n = 0;
        bool hasB = false;
        if (!next_nb(k, n, hasB)) break;
        if (!(ok = wait(bQFull, it) && wait(bKFull0 + gt % Ly::kKStages, gt / Ly::kKStages))) break;
        tc_fence_after();
        issue_s(0, gt);
        if (hasB) issue_s(1, gt);
        mma_commit(BAR(bKEmpty0 + gt % Ly::kKStages));
        if (n == 1) mma_commit(BAR(bQFree));
        for (int j = 0; j < n; ++j) {
          const int g = gt + j;
          const bool more = j + 1 < n;
          ok = wait(bPA, g) && (j > 0 || it == 0 || wait(bOFreeA, it - 1)) &&
               wait(bVFull0 + g % Ly::kVStages, g / Ly::kVStages);
          if (!ok) break;
          tc_fence_after();
          issue_pv(0, g, j > 0);
          if (!more) mma_commit(BAR(bPvA));  // side A's O products of the item are issued
          if (more) {
            if (!(ok = wait(bKFull0 + (g + 1) % Ly::kKStages, (g + 1) / Ly::kKStages))) break;
            tc_fence_after();
            issue_s(0, g + 1);
          }
          if (hasB) {
            if (!(ok = wait(bPB, gB + j) && (j > 0 || itB == 0 || wait(bOFreeB, itB - 1)))) break;
            tc_fence_after();
            issue_pv(1, g, j > 0);
            if (more) issue_s(1, g + 1);
          }
          if (!more && hasB) mma_commit(BAR(bPvB));
          mma_commit(BAR(bVEmpty0 + g % Ly::kVStages));
          if (more) mma_commit(BAR(bKEmpty0 + (g + 1) % Ly::kKStages));
          if (j + 2 == n) mma_commit(BAR(bQFree));  // the item's last S products are issued
        }
        if (!ok) break;
        gt += n;
        ++it;
        if (hasB) {
          gB += n;
          ++itB;
        }
      }
      mma_commit(BAR(bDrain));
      mbar_wait(BAR(bDrain), 0, kWaitNs);
    }
    __syncwarp();
  }
  } else if (warp < kProducerWarp) {
    // ------------------------------------------------------------ softmax A / B
    regs_increase<kSoftmaxRegs>();
    const int side = warp >> 2;  // 0: A (warps 0-3), 1: B (warps 4-7)
    const int r = threadIdx.x - side * 128;  // query row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + side * 128 + lane_off;
    const uint32_t tO = tmem + 256 + side * 128 + lane_off;
    int gx = 0;  // tiles this side has processed
    int ix = 0;  // items this side has processed
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Item I;
      if (!next_item(k, I, true)) {
        if (side == 0 && r == 0) *epi_total = ix;  // no more items: the epilogue stops after ix - 1
        break;
      }
      if (side == 1 && I.h[1] < 0) continue;
      const int i = I.i0 + (I.pk ? (r & (kM / 2 - 1)) : r);  // this row's query token
      const int lim = kCasc ? I.kv_end - 1 : I.c + i;  // last key position this row sees
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < I.n; ++j) {
        // S_j ready; its commit also covers this side's earlier products, so
        // the P columns and O may be rewritten below.
        if (!(ok = wait_w(side ? bSB : bSA, gx + j))) break;
        tc_fence_after();
        int key0, key_end;
        tile_keys(I, j, kFused, key0, key_end, kCasc);
        const bool full = key0 + kN - 1 <= lim && key0 + kN <= key_end;
        uint32_t sr[128];
        tmem_ld64(tS, *reinterpret_cast<uint32_t(*)[64]>(sr));
        tmem_ld64(tS + 64, *reinterpret_cast<uint32_t(*)[64]>(sr + 64));
        tmem_wait_ld();
        // Row maximum of the raw scores (scale > 0, so it commutes with the
        // scaling); masked keys become -inf.
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        // max over the 8-column block starting at column e8
        auto block_max = [&](int e8) {
          const int q = (e8 >> 3) & 3;
          mx[q] = max3(mx[q], __uint_as_float(sr[e8]), __uint_as_float(sr[e8 + 1]));
          mx[q] = max3(mx[q], __uint_as_float(sr[e8 + 2]), __uint_as_float(sr[e8 + 3]));
          mx[q] = max3(mx[q], __uint_as_float(sr[e8 + 4]), __uint_as_float(sr[e8 + 5]));
          mx[q] = max3(mx[q], __uint_as_float(sr[e8 + 6]), __uint_as_float(sr[e8 + 7]));
        };
        if (!full) {
          const int last = min(lim, key_end - 1) - key0;  // last visible column of this row
#pragma unroll
          for (int e2 = 0; e2 < 128; ++e2)
            if (e2 > last) sr[e2] = __float_as_uint(-INFINITY);
        }
#pragma unroll
        for (int e8 = 0; e8 < 128; e8 += 8) block_max(e8);
        const float mt = fmaxf(max3(mx[0], mx[1], mx[2]), mx[3]) * a.scale_log2;
        const float m_new = mt > m_used + 8.f ? mt : m_used;
        const float ref = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = m_used == -INFINITY ? 0.f : ex2(m_used - ref);
        // P = 2^(s * scale - m), rounded to bf16 and packed in pairs into sr[0..63]
        const uint64_t sc2 = f2(a.scale_log2, a.scale_log2);
        const uint64_t nref2 = f2(-ref, -ref);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};  // four (+0, +0) pair sums
        uint32_t* flat = sr;
        auto block_exp = [&](int e8) {
#pragma unroll
          for (int e2 = e8; e2 < e8 + 8; e2 += 2) {
            const uint64_t x = f2_fma(f2(__uint_as_float(flat[e2]), __uint_as_float(flat[e2 + 1])),
                                      sc2, nref2);
            const float2 xc = f2_split(x);
            const uint64_t pp = f2(ex2(xc.x), ex2(xc.y));
            acc[(e2 >> 1) & 3] = f2_add(acc[(e2 >> 1) & 3], pp);
            const float2 pc = f2_split(pp);
            flat[e2 >> 1] = pack_bf16(pc.x, pc.y);
          }
        };
#pragma unroll
        for (int e8 = 0; e8 < 128; e8 += 8) block_exp(e8);
        const float2 s01 = f2_split(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])));
        l = l * alpha + (s01.x + s01.y);
        tmem_st64(tS, *reinterpret_cast<uint32_t(*)[64]>(sr));
        const bool need = j > 0 && m_new != m_used;
        if (__any_sync(0xffffffffu, need)) {
          const float f = need ? alpha : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + cc * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e2 = 0; e2 < 32; ++e2) o[e2] = __float_as_uint(__uint_as_float(o[e2]) * f);
            tmem_st32(tO + cc * 32, o);
          }
        }
        m_used = m_new;
        const int live = key_end - key0;  // rows [live, 128) of V_j are not keys
        if (side == 0 && live < kN) {
          if (!(ok = wait_w(bVFull0 + (gx + j) % Ly::kVStages, (gx + j) / Ly::kVStages))) break;
          uint8_t* vt = sgen + Ly::kV + ((gx + j) % Ly::kVStages) * Ly::kTile;
          const int chunks = (kN - live) * 128 / 16;
          for (int hf = 0; hf < Ly::kHalves; ++hf) {
            uint4* zp = reinterpret_cast<uint4*>(vt + hf * Ly::kHalf + live * 128);
            for (int x = r; x < chunks; x += 128) zp[x] = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(BAR(side ? bPB : bPA));
      }
      if (!ok) break;
      // Hand the row's sum and reference maximum to the epilogue warps, which
      // wait for this side's last product, normalise O and store it, while
      // this warp goes on to the next item.
      EpiSlot& es = epi[(ix & 1) * 2 + side];
      es.l[r] = l;
      es.m[r] = m_used;
      if (r == 0) es.it = I;
      // Hand-off barriers alternate by item parity: a side cannot finish item
      // k + 2 before the epilogue has released item k's O, so neither barrier
      // runs more than one phase ahead of the epilogue's wait on it.
      mbar_arrive(BAR((side ? bLB0 : bLA0) + (ix & 1)));
      gx += I.n;
      ++ix;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp 12 + q reads TMEM lanes 32q .. 32q + 31 (its query rows) of O.
    // Per item: side A, then side B if the item has one.  O is read 16
    // columns at a time; after the last chunk O is released to the next
    // item's products.  Each thread normalises its row by 1 / l, packs it to
    // bf16 and stores it straight to the output, 16 bytes at a time (these
    // warps are off the softmax's critical path, so they need no staging
    // buffer).  The shared-prefix mode writes fp32 partials (O, m, l).
    regs_decrease<kFused ? kEpiRegsFused : kEpiRegs>();
    const int q4 = warp - kEpiWarp0;
    const int r = q4 * 32 + lane;  // query row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    auto finish = [&](int side, int idx, int t0, int i0, int qn, int head, int pk, int hk) -> bool {
      if (!wait_w(side ? bPvB : bPvA, idx)) return false;
      tc_fence_after();
      const EpiSlot& es = epi[(idx & 1) * 2 + side];
      const float l = es.l[r];
      const uint32_t tO = tmem + 256 + side * 128 + lane_off;
      if constexpr (kCasc) {
        // this query row's partial over the chunk: unnormalised O, its
        // reference m (log2 domain) and sum l, in the chunk's slot (t0)
        const int row = head * kM + r;
        const bool live = row < qn;
        float* dst = nullptr;
        if (live) {
          const int seq = row / a.group;
          const int64_t wr = (static_cast<int64_t>(t0) * a.num_decode + seq) * a.hq + hk * a.group +
                             (row - seq * a.group);
          dst = a.ws_o + wr * D;
          a.ws_ml[wr * 2] = es.m[r];
          a.ws_ml[wr * 2 + 1] = l;
        }
#pragma unroll 1
        for (int cc = 0; cc < D / 16; ++cc) {
          uint32_t o[16];
          tmem_ld16(tO + cc * 16, o);
          tmem_wait_ld();
          if (cc == D / 16 - 1) {
            tc_fence_before();
            mbar_arrive(BAR(side ? bOFreeB : bOFreeA));
          }
          if (live) {
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4)
              reinterpret_cast<float4*>(dst + cc * 16)[c4] =
                  make_float4(__uint_as_float(o[4 * c4]), __uint_as_float(o[4 * c4 + 1]),
                              __uint_as_float(o[4 * c4 + 2]), __uint_as_float(o[4 * c4 + 3]));
          }
        }
        return true;
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const uint64_t inv2 = f2(inv, inv);
      // this row's query token and head (packed: rows 64-127 are the next head)
      const int i = i0 + (pk ? (r & (kM / 2 - 1)) : r);
      const bool live = i < qn;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                            static_cast<int64_t>(t0 + (live ? i : 0)) * a.out_stride +
                            static_cast<int64_t>(head + (pk ? (r >> 6) : 0)) * D;
#pragma unroll 1
      for (int cc = 0; cc < D / 16; ++cc) {  // 16-column chunks
        uint32_t o[16];
        tmem_ld16(tO + cc * 16, o);
        tmem_wait_ld();
        if (cc == D / 16 - 1) {
          tc_fence_before();
          mbar_arrive(BAR(side ? bOFreeB : bOFreeA));
        }
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 on =
              f2_split(f2_mul(f2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), inv2));
          w[e] = pack_bf16(on.x, on.y);
        }
        if (live) st_global_v8(orow + cc * 16, w);  // 32 bytes, one instruction
      }
      return true;
    };
    // Wait for side A's hand-off of item ie (1), or learn that side A has no
    // more items (0); -1: the wait ran out or the CTA gave up.  The stop word
    // is looked at between suspending tries, and the warp takes the outcome
    // together.
    auto next_handoff = [&](int ie) -> bool {
      const uint32_t bar = BAR(bLA0 + (ie & 1));
      const uint32_t par = static_cast<uint32_t>(ie >> 1) & 1u;
      const uint64_t limit = a.wait_ns ? a.wait_ns : kWaitNs;
      const uint64_t t0 = globaltimer_ns();
      int res;
      while (true) {
        if (kPoll ? mbar_test_wait(bar, par) : mbar_try_wait(bar, par)) { res = 1; break; }
        if (*epi_total <= ie || *abort_flag) { res = 0; break; }
        if (globaltimer_ns() - t0 > limit) { give_up(); res = 0; break; }
      }
      return __all_sync(0xffffffffu, res == 1);
    };
    int ie = 0, ieB = 0;
    for (;;) {
      if (!next_handoff(ie)) break;
      const Item& I = epi[(ie & 1) * 2].it;
      const int t0 = I.t0, i0 = I.i0, qn = I.qn, hA = I.h[0], hB = I.h[1], pk = I.pk, hk = I.hk;
      if (!finish(0, ie, t0, i0, qn, hA, pk, hk)) break;
      if (hB >= 0) {
        if (!wait_w(bLB0 + (ieB & 1), ieB >> 1) || !finish(1, ieB, t0, i0, qn, hB, pk, hk)) break;
        ++ieB;
      }
      ++ie;
    }
  }
#undef BAR
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- host side -----------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool encode_q(CUtensorMap* m, const AttnArgs& a, int rows = kM) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.hq) * a.head_dim,
                              static_cast<cuuint64_t>(a.num_tokens)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.q_stride) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(rows)};
  const cuuint32_t es[2] = {1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.q), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_cache(CUtensorMap* m, const void* ptr, const AttnArgs& a) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const int bs = 1 << a.bs_log2;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.head_dim), static_cast<cuuint64_t>(a.hkv),
                              static_cast<cuuint64_t>(a.num_blocks) * bs};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.head_dim) * 2,
                                 static_cast<cuuint64_t>(a.hkv) * a.head_dim * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(bs < kN ? bs : kN)};
  const cuuint32_t es[3] = {1, 1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_out(CUtensorMap* m, const AttnArgs& a) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.hq) * a.head_dim,
                              static_cast<cuuint64_t>(a.num_tokens)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.out_stride) * 2};
  const cuuint32_t box[2] = {64, 32};
  const cuuint32_t es[2] = {1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.out, dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q as [tokens, heads, D] with boxes of g heads of one token: the g query
// heads of a kv head, one decode token (cascade prefix pass).
bool encode_q_casc(CUtensorMap* m, const AttnArgs& a) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.head_dim), static_cast<cuuint64_t>(a.hq),
                              static_cast<cuuint64_t>(a.num_tokens)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.head_dim) * 2,
                                 static_cast<cuuint64_t>(a.q_stride) * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(a.group), 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The new tokens' K or V ([T, Hkv, D], token stride in elements): 128-row boxes.
bool encode_new(CUtensorMap* m, const void* ptr, int64_t stride, const AttnArgs& a) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.hkv) * a.head_dim,
                              static_cast<cuuint64_t>(a.num_tokens)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride) * 2};
  const cuuint32_t box[2] = {64, kN};
  const cuuint32_t es[2] = {1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A new work-queue tag for each launch (never 0, so that a zeroed header
// reads as another launch's).
uint32_t next_sched_tag() {
  static std::atomic<uint32_t> tag{0};
  uint32_t t;
  do {
    t = tag.fetch_add(1u, std::memory_order_relaxed) + 1u;
  } while (t == 0u);
  return t;
}

// Highest cost level: every visible key range is at most max_seq_len keys.
int max_level_of(const AttnArgs& a) { return (a.max_seq_len + kN - 1) / kN + 1; }

int64_t total_slots_of(const AttnArgs& a) {
  const int64_t pairs = (a.group + 1) / 2;
  return static_cast<int64_t>(a.hkv) * pairs * (a.num_seqs - a.num_decode) * max_level_of(a);
}

// Lets each instantiation use the layout's dynamic shared memory (once per
// device and instantiation).
template <typename K>
cudaError_t allow_smem(K kernel, int bytes, bool (&done)[64]) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && done[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev < 64) done[dev] = true;
  return e;
}

template <int D, bool kFused>
cudaError_t launch_tc_d(const AttnArgs& args, cudaStream_t st) {
  AttnArgs a = args;
  a.sched_tag = next_sched_tag();
  using Ly = PpLayout<D>;
  static bool done[2][64] = {};
  auto kernel = a.wait_ns ? prefill_tc_kernel<D, kFused, false, true> : prefill_tc_kernel<D, kFused>;
  cudaError_t e = allow_smem(kernel, Ly::kAlloc, done[a.wait_ns ? 1 : 0]);
  if (e != cudaSuccess) return e;
  CUtensorMap mq, mk, mv, mo, mkn, mvn, mq64;
  memset(&mkn, 0, sizeof(mkn));  // unused without the fused scatter
  memset(&mvn, 0, sizeof(mvn));
  if (!encode_q(&mq, a) || !encode_q(&mq64, a, kM / 2) || !encode_cache(&mk, a.k_cache, a) ||
      !encode_cache(&mv, a.v_cache, a) || !encode_out(&mo, a) ||
      (a.k_new && (!encode_new(&mkn, a.k_new, a.kn_stride, a) ||
                   !encode_new(&mvn, a.v_new, a.vn_stride, a))))
    return cudaErrorNotSupported;  // nothing launched: the caller takes the general kernel
  const int total = static_cast<int>(total_slots_of(a));
  int sms = device_num_sms();
  if (a.max_ctas > 0 && a.max_ctas < sms) sms = a.max_ctas;  // SMs left to a concurrent decode
  const int grid = total < sms ? total : sms;
  if (grid <= 0) return cudaSuccess;
  count_launch();
  const int max_level = max_level_of(a);
  e = launch_prio(kernel, dim3(grid), dim3(kThreads), Ly::kAlloc, st,
                  a.has_priority, a.priority, mq, mk, mv, mo, mkn, mvn, mq64, a, total, max_level);
  return e != cudaSuccess ? e : cudaGetLastError();
}

int64_t cascade_tc_slots(const AttnArgs& a) {
  const int64_t tiles = (static_cast<int64_t>(a.num_decode) * a.group + kM - 1) / kM;
  return static_cast<int64_t>(a.hkv) * ((tiles + 1) / 2) * a.nsplit_prefix;
}

template <int D>
cudaError_t launch_casc_d(const AttnArgs& args, cudaStream_t st) {
  AttnArgs a = args;
  a.sched_tag = next_sched_tag();
  using Ly = PpLayout<D>;
  static bool done[2][64] = {};
  auto kernel = a.wait_ns ? prefill_tc_kernel<D, false, true, true> : prefill_tc_kernel<D, false, true>;
  cudaError_t e = allow_smem(kernel, Ly::kAlloc, done[a.wait_ns ? 1 : 0]);
  if (e != cudaSuccess) return e;
  CUtensorMap mq, mk, mv, mo, mkn, mvn, mq64;
  memset(&mkn, 0, sizeof(mkn));
  memset(&mvn, 0, sizeof(mvn));
  memset(&mq64, 0, sizeof(mq64));  // no packed tiles in this mode
  if (!encode_q_casc(&mq, a) || !encode_cache(&mk, a.k_cache, a) ||
      !encode_cache(&mv, a.v_cache, a) || !encode_out(&mo, a))
    return cudaErrorNotSupported;
  const int total = static_cast<int>(cascade_tc_slots(a));
  const int sms = device_num_sms();
  const int grid = total < sms ? total : sms;
  if (grid <= 0) return cudaSuccess;
  count_launch();
  e = launch_prio(kernel, dim3(grid), dim3(kThreads), Ly::kAlloc, st,
                  a.has_priority, a.priority, mq, mk, mv, mo, mkn, mvn, mq64, a, total, 1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool cascade_tc_supported(const AttnArgs& a) {
  const char* env = getenv("PA_CASCADE_IMPL");
  if (env && strcmp(env, "mma") == 0) return false;
  // a kv head's g query heads of one token fill whole 8-row swizzle atoms
  if (a.group % 8 != 0 || a.group > kM || kM % a.group != 0) return false;
  if (static_cast<int64_t>(a.num_decode) * a.group > INT_MAX / 4) return false;
  return prefill_tc_supported(a);
}

cudaError_t launch_cascade_tc(const AttnArgs& a, cudaStream_t st) {
  if (a.num_decode <= 0 || a.nsplit_prefix <= 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_casc_d<128>(a, st) : launch_casc_d<64>(a, st);
}

bool prefill_tc_supported(const AttnArgs& a) {
  const char* env = getenv("PA_PREFILL_IMPL");
  if (env && strcmp(env, "mma") == 0) return false;
  if (a.head_dim != 64 && a.head_dim != 128) return false;
  if (!(a.scale_log2 > 0.f)) return false;  // the row maximum is taken before scaling
  // 16-byte rows for TMA; the epilogue stores 32 bytes at a time
  if ((a.q_stride * 2) % 16 != 0 || (a.out_stride * 2) % 32 != 0) return false;
  if (reinterpret_cast<uintptr_t>(a.out) & 31u) return false;
  if ((reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.k_cache) |
       reinterpret_cast<uintptr_t>(a.v_cache) | reinterpret_cast<uintptr_t>(a.out)) & 15u)
    return false;
  if (total_slots_of(a) > INT_MAX / 2) return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const AttnArgs& a, cudaStream_t st) {
  if (a.num_seqs - a.num_decode <= 0 || a.max_query_len <= 0) return cudaSuccess;
  if (a.k_new) return a.head_dim == 128 ? launch_tc_d<128, true>(a, st) : launch_tc_d<64, true>(a, st);
  return a.head_dim == 128 ? launch_tc_d<128, false>(a, st) : launch_tc_d<64, false>(a, st);
}

}  // namespace pa
