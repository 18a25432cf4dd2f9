// Ragged causal attention for rows with any number of new tokens (prefill and
// chunked prefill), on mma.sync tensor-core tiles.  This is the general path:
// any head_dim in {64, 128}, any power-of-two block size, any GQA ratio.  The
// tcgen05 kernel (prefill_tc.cu) takes over whenever it supports the call
// (scale > 0, 16-byte aligned q rows, 32-byte aligned output rows);
// PA_PREFILL_IMPL=mma forces this one.
//
// Work unit: one CTA per (64-row query tile, kv head, sequence).  The rows of
// a sequence's tile are (new token i, query head of the kv head's group)
// pairs, token-major, so the g query heads that share a kv head share every
// K/V tile.  Keys stream in 64-token chunks from the paged cache (each
// position resolved through the sequence's block table, "vLLM Continuous
// Batching：从 Forward Shape 理解两个核心参数" §2.3补充 第二步) into a
// shared-memory ring filled by all 128 threads with cp.async.  Each warp owns
// 16 rows: S = Q K^T and O += P V are bf16 m16n8k16 mma.sync with fp32
// accumulators, with an online softmax in between.  Token i of a sequence with
// c cached tokens sits at position c + i and sees keys 0 .. c + i of its own
// sequence only (bottom-right aligned causal mask, "vLLM 原理" §3.7: the new
// queries attend to the whole cached sequence).  Tiles are issued heaviest
// first (last rows of each sequence at blockIdx.x = 0).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pa {

namespace {

constexpr int kThreads = 128;
constexpr int kRows = 64;  // query rows per CTA (16 per warp)
constexpr int kKeys = 64;  // keys per chunk

template <int D, int STAGES>
struct PreLayout {
  static constexpr int kRow = D * 2;
  static constexpr int kTile = kKeys * kRow;
  static constexpr int kStage = 2 * kTile;
  static constexpr int kBytes = STAGES * kStage;
};

template <int D, int STAGES>
__global__ void __launch_bounds__(kThreads) prefill_kernel(const AttnArgs a) {
  using Ly = PreLayout<D, STAGES>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int s = a.num_decode + blockIdx.z;
  const int hk = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = __ldg(a.qsl + s);
  const int qn = __ldg(a.qsl + s + 1) - t0;
  const int L = __ldg(a.seq_lens + s);
  if (qn <= 0) return;
  if (L < qn || L > (a.max_blocks << a.bs_log2) || qn > a.max_query_len || L > a.max_seq_len ||
      t0 < 0 || t0 + qn > a.num_tokens) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) flag_error(a.err, PA_DEV_BAD_LEN);
    return;
  }
  const int c = L - qn;  // cached tokens before this step's chunk
  const int g = a.group;
  const int nrows = qn * g;
  const int ntiles = (nrows + kRows - 1) / kRows;
  const int tile = ntiles - 1 - static_cast<int>(blockIdx.x);
  if (tile < 0) return;
  const int R0 = tile * kRows;
  const int i_hi = min(qn - 1, (R0 + kRows - 1) / g);
  const int kv_end = c + i_hi + 1;  // keys this tile can see: [0, kv_end)
  const int nchunks = (kv_end + kKeys - 1) / kKeys;

  // this thread's two rows (A: r, B: r + 8 of the warp's 16)
  const int rA = R0 + warp * 16 + (lane >> 2);
  const int rB = rA + 8;
  const int iA = rA / g, iB = rB / g;
  const bool okA = rA < nrows, okB = rB < nrows;
  const int hA = hk * g + (rA - iA * g), hB = hk * g + (rB - iB * g);
  const int limA = c + iA, limB = c + iB;  // last visible key position
  const int warp_last_row = min(R0 + warp * 16 + 15, nrows - 1);
  const int warp_lim = c + warp_last_row / g;

  uint32_t qa[D / 16][4];
  {
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
    const int cq = (lane & 3) * 2;
    const uint32_t* pa_ = reinterpret_cast<const uint32_t*>(
        q + static_cast<int64_t>(t0 + (okA ? iA : 0)) * a.q_stride +
        static_cast<int64_t>(okA ? hA : 0) * D + cq);
    const uint32_t* pb_ = reinterpret_cast<const uint32_t*>(
        q + static_cast<int64_t>(t0 + (okB ? iB : 0)) * a.q_stride +
        static_cast<int64_t>(okB ? hB : 0) * D + cq);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      qa[ks][0] = okA ? __ldg(pa_ + ks * 8) : 0u;
      qa[ks][1] = okB ? __ldg(pb_ + ks * 8) : 0u;
      qa[ks][2] = okA ? __ldg(pa_ + ks * 8 + 4) : 0u;
      qa[ks][3] = okB ? __ldg(pb_ + ks * 8 + 4) : 0u;
    }
  }

  const __nv_bfloat16* kc = static_cast<const __nv_bfloat16*>(a.k_cache);
  const __nv_bfloat16* vc = static_cast<const __nv_bfloat16*>(a.v_cache);
  const int32_t* bt = a.block_tables + static_cast<int64_t>(s) * a.max_blocks;
  const int64_t slot_stride = static_cast<int64_t>(a.hkv) * D;
  const int64_t head_off = static_cast<int64_t>(hk) * D;
  const int bs_mask = (1 << a.bs_log2) - 1;
  const uint32_t sbase = smem_u32(smem);

  auto load_chunk = [&](int ch, int stage) {
    constexpr int CPR = D / 8;
    const uint32_t kdst = sbase + stage * Ly::kStage;
    const uint32_t vdst = kdst + Ly::kTile;
#pragma unroll
    for (int i = 0; i < kKeys * CPR / kThreads; ++i) {
      const int idx = i * kThreads + threadIdx.x;
      const int r = idx / CPR, cc = idx % CPR;
      const int pos = ch * kKeys + r;
      bool ok = pos < kv_end;
      int64_t off = 0;
      if (ok) {
        const int pb = __ldg(bt + (pos >> a.bs_log2));
        if (pb >= 0 && pb < a.num_blocks) {
          off = static_cast<int64_t>((pb << a.bs_log2) + (pos & bs_mask)) * slot_stride + head_off +
                cc * 8;
        } else {
          ok = false;
          if (cc == 0) flag_error(a.err, PA_DEV_BAD_BLOCK);
        }
      }
      cp_async16(kdst + swz(r, cc, Ly::kRow), kc + off, ok);
      cp_async16(vdst + swz(r, cc, Ly::kRow), vc + off, ok);
    }
  };

#pragma unroll
  for (int st = 0; st < STAGES - 1; ++st) {
    if (st < nchunks) load_chunk(st, st);
    cp_async_commit();
  }

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  for (int ch = 0; ch < nchunks; ++ch) {
    {
      const int cn = ch + STAGES - 1;
      if (cn < nchunks) load_chunk(cn, cn % STAGES);
      cp_async_commit();
    }
    cp_async_wait<STAGES - 1>();
    __syncthreads();
    const int key0 = ch * kKeys;
    if (key0 <= warp_lim) {  // otherwise every row of this warp is masked
      const uint32_t kb = sbase + (ch % STAGES) * Ly::kStage;
      const uint32_t vb = kb + Ly::kTile;
      float sc[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int tr = np * 16 + ((lane >> 4) << 3) + (lane & 7);
          const int ck = ks * 2 + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + swz(tr, ck, Ly::kRow), b0, b1, b2, b3);
          mma_bf16(sc[2 * np], qa[ks], b0, b1);
          mma_bf16(sc[2 * np + 1], qa[ks], b2, b3);
        }
      }
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int pos = key0 + nt * 8 + (lane & 3) * 2 + (j & 1);
          const int lim = j < 2 ? limA : limB;
          const bool vis = pos <= lim && pos < kv_end;
          sc[nt][j] = vis ? sc[nt][j] * a.scale_log2 : -INFINITY;
        }
        mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float r0 = mn0 == -INFINITY ? 0.f : mn0;
      const float r1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = ex2(m0 - r0), al1 = ex2(m1 - r1);
      m0 = mn0;
      m1 = mn1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        sc[nt][0] = ex2(sc[nt][0] - r0);
        sc[nt][1] = ex2(sc[nt][1] - r0);
        sc[nt][2] = ex2(sc[nt][2] - r1);
        sc[nt][3] = ex2(sc[nt][3] - r1);
        ps0 += sc[nt][0] + sc[nt][1];
        ps1 += sc[nt][2] + sc[nt][3];
      }
      l0 = l0 * al0 + ps0;
      l1 = l1 * al1 + ps1;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        o[i][0] *= al0;
        o[i][1] *= al0;
        o[i][2] *= al1;
        o[i][3] *= al1;
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t pa[4] = {pack_bf16(sc[2 * kk][0], sc[2 * kk][1]),
                                pack_bf16(sc[2 * kk][2], sc[2 * kk][3]),
                                pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]),
                                pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3])};
#pragma unroll
        for (int dt2 = 0; dt2 < D / 16; ++dt2) {
          const int tr = kk * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
          const int ck = dt2 * 2 + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + swz(tr, ck, Ly::kRow), b0, b1, b2, b3);
          mma_bf16(o[2 * dt2], pa, b0, b1);
          mma_bf16(o[2 * dt2 + 1], pa, b2, b3);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  const float inv0 = okA ? 1.f / l0 : 0.f, inv1 = okB ? 1.f / l1 : 0.f;
  __nv_bfloat16* oa = out + static_cast<int64_t>(t0 + iA) * a.out_stride + static_cast<int64_t>(hA) * D;
  __nv_bfloat16* ob = out + static_cast<int64_t>(t0 + iB) * a.out_stride + static_cast<int64_t>(hB) * D;
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    const int col = i * 8 + (lane & 3) * 2;
    if (okA) *reinterpret_cast<uint32_t*>(oa + col) = pack_bf16(o[i][0] * inv0, o[i][1] * inv0);
    if (okB) *reinterpret_cast<uint32_t*>(ob + col) = pack_bf16(o[i][2] * inv1, o[i][3] * inv1);
  }
}

constexpr int kStages = 2;

template <int D>
cudaError_t launch_prefill_d(const AttnArgs& a, cudaStream_t st) {
  using Ly = PreLayout<D, kStages>;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, kStages>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::kBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int64_t rows = static_cast<int64_t>(a.max_query_len) * a.group;
  const int tiles = static_cast<int>((rows + kRows - 1) / kRows);
  dim3 grid(tiles, a.hkv, a.num_seqs - a.num_decode);
  count_launch();
  prefill_kernel<D, kStages><<<grid, kThreads, Ly::kBytes, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const AttnArgs& a, cudaStream_t st) {
  if (a.num_seqs - a.num_decode <= 0 || a.max_query_len <= 0) return cudaSuccess;
  if (prefill_tc_supported(a)) {
    const cudaError_t e = launch_prefill_tc(a, st);
    if (e != cudaErrorNotSupported) return e;
  }
  return a.head_dim == 128 ? launch_prefill_d<128>(a, st) : launch_prefill_d<64>(a, st);
}

}  // namespace pa
