// Split-KV decode attention (rows with exactly one new token) and the
// cross-split combine.
//
// Work unit: one CTA per (split j, kv head, group of <= 16 query heads, decode
// sequence).  The CTA's key range [j*part, min(L, (j+1)*part)) is cut into
// 16-token groups; warp w takes groups w, w+4, w+8, ... and streams each
// group's K and V rows (one kv head: 16 rows of head_dim bf16) from the paged
// cache into a private STAGES-deep shared-memory ring with 16-byte cp.async,
// resolving every position through the sequence's block table ("vLLM
// Continuous Batching：从 Forward Shape 理解两个核心参数" §2.3补充 第二步).
// The query heads sharing the kv head are the 16 rows of an m16n8k16 tile, so
// q.k and p.v run as bf16 mma.sync with fp32 accumulation; the online softmax
// (running max m, running sum l, rescaled accumulator — "LLM 推理引擎
// Continuous Batching 与 PagedAttention：从 vLLM 原理到生产级部署实战" §3.3) is
// per warp, then the four warps' (m, l, acc) are merged in shared memory.  A
// sequence covered by one split writes its bf16 output directly; otherwise
// the CTA writes (m, l, acc) to the workspace and combine_kernel merges the
// splits with the same rule: m = max_j m_j, l = sum_j l_j 2^(m_j-m),
// o = sum_j acc_j 2^(m_j-m) / l.  Scores live in the log2 domain (scale is
// pre-multiplied by log2 e).  Split boundaries depend only on logical
// positions, so the result does not depend on where blocks sit in the pool.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pa {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kGrp = 16;  // tokens per warp step

// kFp8: the cache holds E4M3 codes.  The ring then stages the 8-bit rows
// (row pitch D + 16 bytes against bank conflicts) and the products run as
// fp16 mma.sync (every E4M3 value is exact in fp16), with the operand
// fragments converted in registers straight from the staged codes:
//  * K: the head dimension is read in a permuted order (the same for q and
//    k, which leaves q.k unchanged) in which each lane's four dims of a
//    16-dim step are four consecutive bytes: dims t * D/4 + 4 * step + j for
//    lane t = lane % 4, so one 32-bit word per step and key;
//  * V: the 8-bit transposing ldmatrix gives each lane four consecutive keys
//    of one dimension; the keys of a group are permuted the same way in P
//    (score column c of n-tile nt is key 4 (c / 2) + 2 nt + c % 2).
template <int D, int STAGES, bool kFp8>
struct DecLayout {
  static constexpr int kRow = D * 2;         // bytes of one token's K (or V) for one head
  static constexpr int kTile = kGrp * kRow;  // K or V of one group (16-bit)
  static constexpr int kRow8 = D + 16;       // staged 8-bit row (padded)
  static constexpr int kTile8 = kGrp * kRow8;
  static constexpr int kStage = kFp8 ? 2 * kTile8 : 2 * kTile;
  static constexpr int kWarp = STAGES * kStage;
  static constexpr int kLoop = kWarps * kWarp;
  static constexpr int kMergeFloats = 32 + 16 * D;  // m[16], l[16], acc[16][D]
  static constexpr int kMerge = kWarps * kMergeFloats * 4;
  static constexpr int kBytes = kLoop > kMerge ? kLoop : kMerge;
};

template <int D, int STAGES, bool kFp8>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const AttnArgs a) {
  using Ly = DecLayout<D, STAGES, kFp8>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int split = blockIdx.x;
  const int nhc = (a.group + 15) >> 4;
  const int hk = blockIdx.y / nhc;
  const int hc = blockIdx.y - hk * nhc;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int t0 = __ldg(a.qsl + s);
  const int qn = __ldg(a.qsl + s + 1) - t0;
  const int L = __ldg(a.seq_lens + s);
  const bool reporter = split == 0 && blockIdx.y == 0 && threadIdx.x == 0;
  if (qn != 1 || t0 < 0 || t0 >= a.num_tokens) {
    if (reporter) flag_error(a.err, qn != 1 ? PA_DEV_BAD_DECODE : PA_DEV_BAD_LEN);
    return;
  }
  if (L < 1 || L > a.max_seq_len || L > (a.max_blocks << a.bs_log2)) {
    if (reporter) flag_error(a.err, PA_DEV_BAD_LEN);
    return;
  }
  // Keys [key_begin, L); key_begin > 0 only in the suffix pass of a cascade,
  // which needs a key of the sequence's own past the shared prefix.
  if (L <= a.key_begin) {
    if (reporter) flag_error(a.err, PA_DEV_BAD_LEN);
    return;
  }
  const int nsplit = (L - a.key_begin + a.part - 1) / a.part;
  if (split >= nsplit) return;
  const int p_lo = a.key_begin + split * a.part;
  const int p_hi = min(L, p_lo + a.part);
  const int ngroups = (p_hi - p_lo + kGrp - 1) / kGrp;
  const int rows = min(16, a.group - hc * 16);  // live query heads in this CTA
  const int h0 = hk * a.group + hc * 16;

  // A fragments of the 16 x D query tile (row = query head); absent heads are 0.
  uint32_t qa[D / 16][4];
  {
    const int r = lane >> 2, cq = (lane & 3) * 2;
    const __nv_bfloat16* qrow =
        static_cast<const __nv_bfloat16*>(a.q) + static_cast<int64_t>(t0) * a.q_stride;
    const bool va = r < rows, vb = r + 8 < rows;
    const uint32_t* pa_ = reinterpret_cast<const uint32_t*>(
        qrow + static_cast<int64_t>(h0 + (va ? r : 0)) * D + cq);
    const uint32_t* pb_ = reinterpret_cast<const uint32_t*>(
        qrow + static_cast<int64_t>(h0 + (vb ? r + 8 : 0)) * D + cq);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      qa[ks][0] = va ? __ldg(pa_ + ks * 8) : 0u;
      qa[ks][1] = vb ? __ldg(pb_ + ks * 8) : 0u;
      qa[ks][2] = va ? __ldg(pa_ + ks * 8 + 4) : 0u;
      qa[ks][3] = vb ? __ldg(pb_ + ks * 8 + 4) : 0u;
    }
    if (kFp8) {
      // permuted dims (see DecLayout): A regs {0,1} = dims t*D/4 + 4ks + {0,1},
      // regs {2,3} = + {2,3}; bf16 -> fp16 pairs (exact in range)
      const uint32_t* qa32 = reinterpret_cast<const uint32_t*>(
          qrow + static_cast<int64_t>(h0 + (va ? r : 0)) * D + (lane & 3) * (D / 4));
      const uint32_t* qb32 = reinterpret_cast<const uint32_t*>(
          qrow + static_cast<int64_t>(h0 + (vb ? r + 8 : 0)) * D + (lane & 3) * (D / 4));
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qa[ks][0] = va ? __ldg(qa32 + 2 * ks) : 0u;
        qa[ks][1] = vb ? __ldg(qb32 + 2 * ks) : 0u;
        qa[ks][2] = va ? __ldg(qa32 + 2 * ks + 1) : 0u;
        qa[ks][3] = vb ? __ldg(qb32 + 2 * ks + 1) : 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&qa[ks][j]);
          qa[ks][j] = pack_f16(__low2float(b), __high2float(b));
        }
      }
    }
  }

  const __nv_bfloat16* kc = static_cast<const __nv_bfloat16*>(a.k_cache);
  const __nv_bfloat16* vc = static_cast<const __nv_bfloat16*>(a.v_cache);
  const int32_t* bt = a.block_tables + static_cast<int64_t>(s) * a.max_blocks;
  const int64_t slot_stride = static_cast<int64_t>(a.hkv) * D;  // elements per cache slot
  const int64_t head_off = static_cast<int64_t>(hk) * D;
  const int bs_mask = (1 << a.bs_log2) - 1;
  const uint32_t wbase = smem_u32(smem) + warp * Ly::kWarp;

  // Stage one 16-token group: lane r < 16 resolves position p + r to its
  // cache slot; every lane then copies D/16 16-byte pieces of K and of V.
  // Positions outside [p_lo, p_hi) or on a bad block are zero-filled.
  auto load_group = [&](int gi, int stage) {
    const int p = p_lo + gi * kGrp;
    int my_slot = -1;
    {
      const int pos = p + (lane & 15);
      if (pos < p_hi) {
        const int pb = __ldg(bt + (pos >> a.bs_log2));
        if (pb >= 0 && pb < a.num_blocks) {
          my_slot = (pb << a.bs_log2) + (pos & bs_mask);
        } else if (lane < 16) {
          flag_error(a.err, PA_DEV_BAD_BLOCK);
        }
      }
    }
    const uint32_t kdst = wbase + stage * Ly::kStage;
    if (kFp8) {
      const uint32_t vdst = kdst + Ly::kTile8;
      const uint8_t* kc8 = static_cast<const uint8_t*>(a.k_cache);
      const uint8_t* vc8 = static_cast<const uint8_t*>(a.v_cache);
      constexpr int CPR8 = D / 16;  // 16-byte pieces per 8-bit row
#pragma unroll
      for (int i = 0; i < kGrp * CPR8 / 32; ++i) {
        const int idx = i * 32 + lane;
        const int r = idx / CPR8, c = idx % CPR8;
        const int slot = __shfl_sync(0xffffffffu, my_slot, r);
        const bool ok = slot >= 0;
        const int64_t off = ok ? static_cast<int64_t>(slot) * slot_stride + head_off + c * 16 : 0;
        cp_async16(kdst + r * Ly::kRow8 + c * 16, kc8 + off, ok);
        cp_async16(vdst + r * Ly::kRow8 + c * 16, vc8 + off, ok);
      }
      return;
    }
    const uint32_t vdst = kdst + Ly::kTile;
    constexpr int CPR = D / 8;  // 16-byte pieces per row
#pragma unroll
    for (int i = 0; i < kGrp * CPR / 32; ++i) {
      const int idx = i * 32 + lane;
      const int r = idx / CPR, c = idx % CPR;
      const int slot = __shfl_sync(0xffffffffu, my_slot, r);
      const bool ok = slot >= 0;
      const int64_t off = ok ? static_cast<int64_t>(slot) * slot_stride + head_off + c * 8 : 0;
      cp_async16(kdst + swz(r, c, Ly::kRow), kc + off, ok);
      cp_async16(vdst + swz(r, c, Ly::kRow), vc + off, ok);
    }
  };

  const int my_groups = ngroups > warp ? (ngroups - warp + kWarps - 1) / kWarps : 0;
#pragma unroll
  for (int st = 0; st < STAGES - 1; ++st) {
    if (st < my_groups) load_group(warp + st * kWarps, st);
    cp_async_commit();
  }

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  for (int k = 0; k < my_groups; ++k) {
    {
      const int kn = k + STAGES - 1;
      if (kn < my_groups) load_group(warp + kn * kWarps, kn % STAGES);
      cp_async_commit();
    }
    cp_async_wait<STAGES - 1>();
    __syncwarp();
    const int st = k % STAGES;
    const uint32_t kb = wbase + st * Ly::kStage;
    const uint32_t vb = kb + (kFp8 ? Ly::kTile8 : Ly::kTile);
    const int p = p_lo + (warp + k * kWarps) * kGrp;

    const bool full = p + kGrp <= p_hi;  // no key of the group is past the range

    // S (16 heads x 16 tokens) = Q K^T
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if (kFp8) {
      const uint8_t* k8 = smem + (kb - smem_u32(smem));
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int n = lane >> 2;
        const int key = 4 * (n >> 1) + 2 * nt + (n & 1);
        const uint4* row = reinterpret_cast<const uint4*>(k8 + key * Ly::kRow8 + (lane & 3) * (D / 4));
        uint32_t w[D / 16];
#pragma unroll
        for (int x = 0; x < D / 64; ++x) {
          const uint4 v4 = row[x];
          w[4 * x] = v4.x;
          w[4 * x + 1] = v4.y;
          w[4 * x + 2] = v4.z;
          w[4 * x + 3] = v4.w;
        }
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t b0, b1;
          cvt_e4m3x4_f16(w[ks], b0, b1);
          mma_f16(sc[nt], qa[ks], b0, b1);
        }
      }
    } else {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int tr = ((lane >> 4) << 3) + (lane & 7);
        const int ck = ks * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + swz(tr, ck, Ly::kRow), b0, b1, b2, b3);
        mma_bf16(sc[0], qa[ks], b0, b1);
        mma_bf16(sc[1], qa[ks], b2, b3);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int pos = kFp8 ? p + 4 * (lane & 3) + 2 * nt + (j & 1)
                             : p + nt * 8 + (lane & 3) * 2 + (j & 1);
        sc[nt][j] = full || pos < p_hi ? sc[nt][j] * a.scale_log2 : -INFINITY;
      }
    float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
    float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    // The running max only moves when the group's max exceeds it by more than
    // 8 (a factor 256): P then stays <= 256, and the numerator and the sum use
    // the same reference, so the result does not depend on it.  O is rescaled
    // only when some row's reference moved.
    const float mn0 = mx0 > m0 + 8.f ? mx0 : m0, mn1 = mx1 > m1 + 8.f ? mx1 : m1;
    const bool moved = __any_sync(0xffffffffu, mn0 != m0 || mn1 != m1);
    const float r0 = mn0 == -INFINITY ? 0.f : mn0;
    const float r1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = ex2(m0 - r0), al1 = ex2(m1 - r1);
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      sc[nt][0] = ex2(sc[nt][0] - r0);
      sc[nt][1] = ex2(sc[nt][1] - r0);
      sc[nt][2] = ex2(sc[nt][2] - r1);
      sc[nt][3] = ex2(sc[nt][3] - r1);
    }
    l0 = l0 * al0 + (sc[0][0] + sc[0][1]) + (sc[1][0] + sc[1][1]);
    l1 = l1 * al1 + (sc[0][2] + sc[0][3]) + (sc[1][2] + sc[1][3]);
    if (moved) {
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        o[i][0] *= al0;
        o[i][1] *= al0;
        o[i][2] *= al1;
        o[i][3] *= al1;
      }
    }
    uint32_t pa[4];
    if (kFp8) {
      pa[0] = pack_f16(sc[0][0], sc[0][1]);
      pa[1] = pack_f16(sc[0][2], sc[0][3]);
      pa[2] = pack_f16(sc[1][0], sc[1][1]);
      pa[3] = pack_f16(sc[1][2], sc[1][3]);
    } else {
      pa[0] = pack_bf16(sc[0][0], sc[0][1]);
      pa[1] = pack_bf16(sc[0][2], sc[0][3]);
      pa[2] = pack_bf16(sc[1][0], sc[1][1]);
      pa[3] = pack_bf16(sc[1][2], sc[1][3]);
    }
    // O (16 heads x D) += P V
#pragma unroll
    for (int dt2 = 0; dt2 < D / 16; ++dt2) {
      if (kFp8) {
        // lane: keys 4t .. 4t+3 of dims dt2*16 + lane/4 (r0) and + 8 (r1)
        uint32_t r0, r1, b0, b1, b2, b3;
        ldsm8_t(vb + (lane & 15) * Ly::kRow8 + dt2 * 16, r0, r1);
        cvt_e4m3x4_f16(r0, b0, b1);
        cvt_e4m3x4_f16(r1, b2, b3);
        mma_f16(o[2 * dt2], pa, b0, b1);
        mma_f16(o[2 * dt2 + 1], pa, b2, b3);
      } else {
        const int tr = (((lane >> 3) & 1) << 3) + (lane & 7);
        const int ck = dt2 * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swz(tr, ck, Ly::kRow), b0, b1, b2, b3);
        mma_bf16(o[2 * dt2], pa, b0, b1);
        mma_bf16(o[2 * dt2 + 1], pa, b2, b3);
      }
    }
    __syncwarp();
  }

  // merge the four warps' partial softmax states
  cp_async_wait<0>();
  __syncthreads();
  float* ms = reinterpret_cast<float*>(smem);
  {
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    float* mw = ms + warp * Ly::kMergeFloats;
    const int r = lane >> 2;
    if ((lane & 3) == 0) {
      mw[r] = m0;
      mw[r + 8] = m1;
      mw[16 + r] = l0;
      mw[16 + r + 8] = l1;
    }
    float* ow = mw + 32;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      const int c = i * 8 + (lane & 3) * 2;
      ow[r * D + c] = o[i][0];
      ow[r * D + c + 1] = o[i][1];
      ow[(r + 8) * D + c] = o[i][2];
      ow[(r + 8) * D + c + 1] = o[i][3];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < rows * D; idx += kThreads) {
    const int rr = idx / D, d = idx - rr * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ms[w * Ly::kMergeFloats + rr]);
    float lsum = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float* mw = ms + w * Ly::kMergeFloats;
      const float mv = mw[rr];
      const float wt = mv == -INFINITY ? 0.f : ex2(mv - M);
      lsum += wt * mw[16 + rr];
      acc += wt * mw[32 + rr * D + d];
    }
    if (kFp8) lsum *= a.inv_v_scale;  // out = acc * v_scale / l
    const int h = h0 + rr;
    if (nsplit == 1 && !a.cascade) {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
      out[static_cast<int64_t>(t0) * a.out_stride + static_cast<int64_t>(h) * D + d] =
          __float2bfloat16_rn(acc / lsum);
    } else {
      const int64_t row = (static_cast<int64_t>(a.split0 + split) * a.num_decode + s) * a.hq + h;
      a.ws_o[row * D + d] = acc;
      if (d == 0) {
        a.ws_ml[row * 2] = M;
        a.ws_ml[row * 2 + 1] = lsum;
      }
    }
  }
}

// One warp per (decode sequence, query head): merge that row's splits.
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const AttnArgs a) {
  const int s = blockIdx.x;
  const int h = blockIdx.y * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (h >= a.hq) return;
  const int t0 = __ldg(a.qsl + s);
  const int qn = __ldg(a.qsl + s + 1) - t0;
  const int L = __ldg(a.seq_lens + s);
  if (qn != 1 || t0 < 0 || t0 >= a.num_tokens || L < 1 || L > a.max_seq_len ||
      L > (a.max_blocks << a.bs_log2))
    return;
  if (L <= a.key_begin) return;
  // prefix partials (cascade) first, then this row's splits of [key_begin, L)
  const int n = a.nsplit_prefix + (L - a.key_begin + a.part - 1) / a.part;
  if (n <= 1) return;
  const int64_t stride = static_cast<int64_t>(a.num_decode) * a.hq;
  const int64_t row0 = static_cast<int64_t>(s) * a.hq + h;
  // One pass with a running maximum, four partials at a time so that their
  // loads are in flight together (the merge is exact in any order).
  float M = -INFINITY, lsum = 0.f;
  float acc[D / 32];
#pragma unroll
  for (int i = 0; i < D / 32; ++i) acc[i] = 0.f;
  for (int j0 = 0; j0 < n; j0 += 4) {
    float mj[4], lj[4], oj[4][D / 32];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool live = j0 + u < n;
      const int64_t row = row0 + static_cast<int64_t>(live ? j0 + u : j0) * stride;
      mj[u] = live ? a.ws_ml[row * 2] : -INFINITY;
      lj[u] = live ? a.ws_ml[row * 2 + 1] : 0.f;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) oj[u][i] = live ? a.ws_o[row * D + lane + 32 * i] : 0.f;
    }
    const float Mn = fmaxf(fmaxf(M, fmaxf(mj[0], mj[1])), fmaxf(mj[2], mj[3]));
    const float c = M == -INFINITY ? 0.f : ex2(M - Mn);
    lsum *= c;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[i] *= c;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = mj[u] == -INFINITY ? 0.f : ex2(mj[u] - Mn);
      lsum += w * lj[u];
#pragma unroll
      for (int i = 0; i < D / 32; ++i) acc[i] += w * oj[u][i];
    }
    M = Mn;
  }
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + static_cast<int64_t>(t0) * a.out_stride +
                       static_cast<int64_t>(h) * D;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) out[lane + 32 * i] = __float2bfloat16_rn(acc[i] / lsum);
}

template <int D>
cudaError_t launch_combine_d(const AttnArgs& a, cudaStream_t st) {
  count_launch();
  cudaError_t e = launch_prio(combine_kernel<D>, dim3(a.num_decode, (a.hq + 3) / 4), dim3(128), 0,
                              st, a.has_priority, a.priority, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

constexpr int kStages = 3;
constexpr int kStages8 = 4;  // 8-bit stages are half the bytes: one more in flight

template <int D, bool kFp8>
cudaError_t launch_decode_d(const AttnArgs& a, cudaStream_t st) {
  constexpr int kSt = kFp8 ? kStages8 : kStages;
  using Ly = DecLayout<D, kSt, kFp8>;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, kSt, kFp8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::kBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int nhc = (a.group + 15) / 16;
  dim3 grid(a.nsplit, a.hkv * nhc, a.num_decode);
  count_launch();
  cudaError_t e = launch_prio(decode_kernel<D, kSt, kFp8>, grid, dim3(kThreads), Ly::kBytes, st,
                              a.has_priority, a.priority, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess || (a.nsplit <= 1 && !a.cascade) || a.defer_combine) return e;
  return launch_combine_d<D>(a, st);
}

}  // namespace

void decode_partition(int num_decode, int hkv_units, int max_seq_len, int num_sms, int* part,
                      int* nsplit) {
  // Enough CTAs for several waves at two CTAs per SM, but never splits
  // shorter than 256 tokens (the combine pass must stay negligible).
  const int64_t base = static_cast<int64_t>(num_decode) * hkv_units;
  const int64_t want = static_cast<int64_t>(num_sms) * 8;
  int n = base > 0 ? static_cast<int>((want + base - 1) / base) : 1;
  const int max_n = max_seq_len > 256 ? (max_seq_len + 255) / 256 : 1;
  if (n > max_n) n = max_n;
  if (n < 1) n = 1;
  int p = (max_seq_len + n - 1) / n;
  p = ((p + 63) / 64) * 64;
  if (p < 64) p = 64;
  *part = p;
  *nsplit = (max_seq_len + p - 1) / p;
  if (*nsplit < 1) *nsplit = 1;
}

cudaError_t launch_combine(const AttnArgs& a, cudaStream_t st) {
  if (a.num_decode <= 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_combine_d<128>(a, st) : launch_combine_d<64>(a, st);
}

cudaError_t launch_decode(const AttnArgs& a, cudaStream_t st) {
  if (a.num_decode <= 0) return cudaSuccess;
  if (a.kv_fp8)
    return a.head_dim == 128 ? launch_decode_d<128, true>(a, st) : launch_decode_d<64, true>(a, st);
  return a.head_dim == 128 ? launch_decode_d<128, false>(a, st) : launch_decode_d<64, false>(a, st);
}

}  // namespace pa
