// Shared-prefix ("cascade") decode attention: the prefix pass.
//
// Requests that share a prompt share its cached blocks ("vLLM 原理" §2.3
// Automatic Prefix Cache; §2.1 copy-on-write keeps the shared blocks
// read-only).  When every decode sequence of a step starts with the same P
// key positions (the same physical blocks), the split-KV decode kernel would
// read those P keys once per sequence.  This pass reads them once per group
// of 128 query rows instead: for every (decode sequence, query head) row it
// computes the online-softmax partial (m, l, acc) over the prefix keys.  The
// decode kernel then covers each sequence's own keys [P, L), and the combine
// merges both with the split-KV merge (m = max_j m_j,
// l = sum_j l_j 2^(m_j - m), o = sum_j acc_j 2^(m_j - m) / l), which is exact
// for any partition of the keys.
//
// CTA: 128 query rows of one kv head (8 warps x 16 rows) and one chunk of the
// prefix; two CTAs per SM (128 registers a thread).  Row r of a kv head's rows is (decode sequence r / g, query head
// hk * g + r % g), g = query heads per kv head.  The chunk's keys stream
// through a 3-stage ring of 32-key stages (the kv head's K and V rows, 16-byte
// cp.async by all threads, block ids from the first sequence's table); every
// warp runs each stage against its own 16 rows: q.k and p.v as m16n8k16 bf16
// mma.sync with fp32 accumulation, scores in the log2 domain, and a running
// max that only moves when a group's max exceeds it by more than 8.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pa {

namespace {

constexpr int kCWarps = 8;
constexpr int kCThreads = kCWarps * 32;
constexpr int kCRows = kCWarps * 16;  // query rows per CTA
constexpr int kCKeys = 32;            // keys per stage
constexpr int kCStages = 3;

template <int D>
struct CascLayout {
  static constexpr int kRow = D * 2;           // bytes of one key's K (or V) for one head
  static constexpr int kTile = kCKeys * kRow;  // K or V of one stage
  static constexpr int kStage = 2 * kTile;
  static constexpr int kBytes = kCStages * kStage;
};

template <int D>
__global__ void __launch_bounds__(kCThreads, 2) cascade_prefix_kernel(const AttnArgs a) {
  using Ly = CascLayout<D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int split = blockIdx.x;
  const int hk = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = a.group;
  const int nrows = a.num_decode * g;  // query rows of one kv head
  const int k_lo = split * a.part_prefix;
  const int k_hi = min(a.prefix_len, k_lo + a.part_prefix);
  if (k_lo >= k_hi) return;
  const int nst = (k_hi - k_lo + kCKeys - 1) / kCKeys;

  // This lane's two rows (r = lane / 4 and r + 8 of the warp's 16): the
  // sequence, the query head and whether the row is a valid decode row whose
  // keys extend past the prefix (others are left to the decode kernel, which
  // reports them, and get no partial).
  int seq[2], head[2];
  bool valid[2];
  uint32_t qa[D / 16][4];
  {
    const int cq = (lane & 3) * 2;
    const uint32_t* qp[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int row = blockIdx.z * kCRows + warp * 16 + (lane >> 2) + hh * 8;
      bool ok = row < nrows;
      const int sq = ok ? row / g : 0;
      const int h = hk * g + (ok ? row - sq * g : 0);
      int t0 = 0;
      if (ok) {
        t0 = __ldg(a.qsl + sq);
        const int qn = __ldg(a.qsl + sq + 1) - t0;
        const int L = __ldg(a.seq_lens + sq);
        ok = qn == 1 && t0 >= 0 && t0 < a.num_tokens && L > a.prefix_len && L <= a.max_seq_len &&
             L <= (a.max_blocks << a.bs_log2);
        if (!ok) t0 = 0;
      }
      seq[hh] = sq;
      head[hh] = h;
      valid[hh] = ok;
      qp[hh] = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                 static_cast<int64_t>(t0) * a.q_stride +
                                                 static_cast<int64_t>(h) * D + cq);
    }
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      qa[ks][0] = valid[0] ? __ldg(qp[0] + ks * 8) : 0u;
      qa[ks][1] = valid[1] ? __ldg(qp[1] + ks * 8) : 0u;
      qa[ks][2] = valid[0] ? __ldg(qp[0] + ks * 8 + 4) : 0u;
      qa[ks][3] = valid[1] ? __ldg(qp[1] + ks * 8 + 4) : 0u;
    }
  }

  const __nv_bfloat16* kc = static_cast<const __nv_bfloat16*>(a.k_cache);
  const __nv_bfloat16* vc = static_cast<const __nv_bfloat16*>(a.v_cache);
  const int32_t* bt = a.block_tables;  // the prefix blocks are the same in every table
  const int64_t slot_stride = static_cast<int64_t>(a.hkv) * D;
  const int64_t head_off = static_cast<int64_t>(hk) * D;
  const int bs_mask = (1 << a.bs_log2) - 1;
  const uint32_t sbase = smem_u32(smem);

  // Stage `si` of the chunk (keys k_lo + 64 si ...) into ring slot `slot`:
  // every thread copies 16-byte pieces of K and V; keys past the chunk or on
  // a bad block are zero-filled.
  auto load_stage = [&](int si, int slot) {
    constexpr int CPR = D / 8;  // 16-byte pieces per row
    const uint32_t kdst = sbase + slot * Ly::kStage;
    const uint32_t vdst = kdst + Ly::kTile;
#pragma unroll
    for (int i = 0; i < kCKeys * CPR / kCThreads; ++i) {
      const int idx = i * kCThreads + threadIdx.x;
      const int r = idx / CPR, c = idx % CPR;
      const int pos = k_lo + si * kCKeys + r;
      bool ok = pos < k_hi;
      int64_t off = 0;
      if (ok) {
        const int pb = __ldg(bt + (pos >> a.bs_log2));
        ok = pb >= 0 && pb < a.num_blocks;
        if (ok) {
          off = static_cast<int64_t>((pb << a.bs_log2) + (pos & bs_mask)) * slot_stride + head_off +
                c * 8;
        } else if (c == 0) {
          flag_error(a.err, PA_DEV_BAD_BLOCK);
        }
      }
      cp_async16(kdst + swz(r, c, Ly::kRow), kc + off, ok);
      cp_async16(vdst + swz(r, c, Ly::kRow), vc + off, ok);
    }
  };

#pragma unroll
  for (int st = 0; st < kCStages - 1; ++st) {
    if (st < nst) load_stage(st, st);
    cp_async_commit();
  }

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  for (int k = 0; k < nst; ++k) {
    {
      const int kn = k + kCStages - 1;
      if (kn < nst) load_stage(kn, kn % kCStages);
      cp_async_commit();
    }
    cp_async_wait<kCStages - 1>();
    __syncthreads();
    const uint32_t kb = sbase + (k % kCStages) * Ly::kStage;
    const uint32_t vb = kb + Ly::kTile;
#pragma unroll 1
    for (int sub = 0; sub < kCKeys / 16; ++sub) {
      const int p = k_lo + k * kCKeys + sub * 16;
      if (p >= k_hi) break;
      const bool full = p + 16 <= k_hi;
      // S (16 rows x 16 keys) = Q K^T
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int tr = sub * 16 + ((lane >> 4) << 3) + (lane & 7);
        const int ck = ks * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + swz(tr, ck, Ly::kRow), b0, b1, b2, b3);
        mma_bf16(sc[0], qa[ks], b0, b1);
        mma_bf16(sc[1], qa[ks], b2, b3);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int pos = p + nt * 8 + (lane & 3) * 2 + (j & 1);
          sc[nt][j] = full || pos < k_hi ? sc[nt][j] * a.scale_log2 : -INFINITY;
        }
      float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
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
      pa[0] = pack_bf16(sc[0][0], sc[0][1]);
      pa[1] = pack_bf16(sc[0][2], sc[0][3]);
      pa[2] = pack_bf16(sc[1][0], sc[1][1]);
      pa[3] = pack_bf16(sc[1][2], sc[1][3]);
      // O (16 rows x D) += P V
#pragma unroll
      for (int dt2 = 0; dt2 < D / 16; ++dt2) {
        const int tr = sub * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
        const int ck = dt2 * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swz(tr, ck, Ly::kRow), b0, b1, b2, b3);
        mma_bf16(o[2 * dt2], pa, b0, b1);
        mma_bf16(o[2 * dt2 + 1], pa, b2, b3);
      }
    }
    __syncthreads();  // the slot is refilled in the next iteration
  }
  cp_async_wait<0>();

  // Partial of each valid row into prefix slot `split`.
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    if (!valid[hh]) continue;
    const int64_t row = (static_cast<int64_t>(split) * a.num_decode + seq[hh]) * a.hq + head[hh];
    float* dst = a.ws_o + row * D + (lane & 3) * 2;
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
      *reinterpret_cast<float2*>(dst + i * 8) = make_float2(o[i][2 * hh], o[i][2 * hh + 1]);
    if ((lane & 3) == 0) {
      a.ws_ml[row * 2] = hh ? m1 : m0;
      a.ws_ml[row * 2 + 1] = hh ? l1 : l0;
    }
  }
}

template <int D>
cudaError_t launch_cascade_d(const AttnArgs& a, cudaStream_t st) {
  using Ly = CascLayout<D>;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(cascade_prefix_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::kBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int tiles = (a.num_decode * a.group + kCRows - 1) / kCRows;
  dim3 grid(a.nsplit_prefix, a.hkv, tiles);
  count_launch();
  cudaError_t e = launch_prio(cascade_prefix_kernel<D>, grid, dim3(kCThreads), Ly::kBytes, st,
                              a.has_priority, a.priority, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

void cascade_partition(int num_decode, int hq, int hkv, int prefix_len, int num_sms, bool tc,
                       int* part_prefix, int* nsplit_prefix) {
  if (tc) {
    // Tensor-core pass: items of (kv head, pair of 128-row tiles, chunk) on a
    // persistent grid of one CTA per SM.  Chunks are whole 128-key tiles; take
    // the count with the shortest estimated makespan (waves of items times
    // tiles per item plus about 1.5 tiles of per-item cost, and a little per
    // chunk for the merge).
    const int group = hkv > 0 ? hq / hkv : 1;
    const int64_t tiles =
        (static_cast<int64_t>(num_decode) * group + 127) / 128;
    const int64_t pairs = static_cast<int64_t>(hkv) * ((tiles + 1) / 2);
    const int ktiles = (prefix_len + 127) / 128;
    const int sms = num_sms > 0 ? num_sms : 1;
    int best = 1;
    double best_t = 1e300;
    for (int n = 1; n <= ktiles && n <= 256; ++n) {
      const int per = (ktiles + n - 1) / n;
      const int64_t items = pairs * ((ktiles + per - 1) / per);
      const double t = static_cast<double>((items + sms - 1) / sms) * (per + 1.5) + 0.05 * n;
      if (t < best_t - 1e-9) {
        best_t = t;
        best = n;
      }
    }
    const int per = (ktiles + best - 1) / best;
    *part_prefix = per * 128;
    *nsplit_prefix = prefix_len > 0 ? (prefix_len + *part_prefix - 1) / *part_prefix : 0;
    return;
  }
  // Chunks of at least 256 keys.  Among the chunk counts that give at least
  // one full wave of CTAs (two per SM), take the one whose last wave is
  // fullest, with a small charge per chunk (each adds a partial per row to
  // merge).
  const int group = hkv > 0 ? hq / hkv : 1;
  const int64_t tiles =
      static_cast<int64_t>(hkv) * ((static_cast<int64_t>(num_decode) * group + kCRows - 1) / kCRows);
  const int64_t slots = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 2;
  const int max_n = prefix_len > 256 ? (prefix_len + 255) / 256 : 1;
  int best = 1;
  double best_score = -1e30;
  for (int n = 1; n <= max_n && n <= 256; ++n) {
    const int p = ((prefix_len + n - 1) / n + kCKeys - 1) / kCKeys * kCKeys;
    const int64_t ctas = tiles * ((prefix_len + p - 1) / p);
    const int64_t waves = (ctas + slots - 1) / slots;
    double score = static_cast<double>(ctas) / static_cast<double>(waves * slots) - 0.002 * n;
    if (ctas < slots) score -= 1.0;  // less than one wave: the SMs are not all busy
    if (score > best_score + 1e-9) {
      best_score = score;
      best = n;
    }
  }
  int p = (prefix_len + best - 1) / best;
  p = ((p + kCKeys - 1) / kCKeys) * kCKeys;
  if (p < kCKeys) p = kCKeys;
  *part_prefix = p;
  *nsplit_prefix = prefix_len > 0 ? (prefix_len + p - 1) / p : 0;
}

cudaError_t launch_cascade_prefix(const AttnArgs& a, cudaStream_t st) {
  if (a.num_decode <= 0 || a.nsplit_prefix <= 0) return cudaSuccess;
  if (a.casc_tc) return launch_cascade_tc(a, st);
  return a.head_dim == 128 ? launch_cascade_d<128>(a, st) : launch_cascade_d<64>(a, st);
}

}  // namespace pa
