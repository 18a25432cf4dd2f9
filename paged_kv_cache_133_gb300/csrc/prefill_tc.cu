// Ragged causal prefill on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Work unit: one CTA per (128-query tile, query head, sequence).  Query token
// i of a sequence with c cached tokens sits at position c + i and sees keys
// 0 .. c + i of its own sequence (bottom-right aligned causal mask; "vLLM 原理"
// §3.7: new queries attend to the whole cached sequence).  Keys are consumed
// in tiles of 128 positions; each tile is gathered from the paged cache by TMA,
// one box per physical block found through the sequence's block table ("vLLM
// Continuous Batching：从 Forward Shape 理解两个核心参数" §2.3补充 第二步).
//
// Warp roles (192 threads):
//   warps 0-3  softmax + epilogue; thread r owns query row r = TMEM lane r
//   warp 4     TMA producer: Q once, then K_j / V_j into a 2-stage ring
//   warp 5     TMEM allocation and MMA issue (one elected lane)
// Per key tile j:
//   S_j = Q K_j^T        tcgen05.mma kind::f16, 128x128x(head_dim), fp32 in TMEM
//                        (two S buffers, so S_{j+1} runs while row j's softmax does)
//   softmax              tcgen05.ld of the row, mask, scale, online max / sum,
//                        P = 2^(s - m) rounded to bf16 into 128B-swizzled smem
//   O += P V_j           tcgen05.mma with V read MN-major; O stays in TMEM
// The running max m only moves when a row's tile maximum exceeds it by more
// than 8 (a factor 256 in the exponent base 2); O and l are then rescaled by
// 2^(m_old - m_new).  Because numerator and denominator use the same m the
// result is exact for any choice of m; the threshold only bounds P <= 256.
// All scores are in the log2 domain (scale pre-multiplied by log2 e).
//
// Every mbarrier wait is bounded (2 s of wall time); on expiry the kernel sets
// PA_DEV_TIMEOUT, lets its in-flight copies and MMAs drain (again bounded),
// frees TMEM and exits.
#include <cuda.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace pa {

namespace {

using namespace tc;

constexpr int kM = 128;  // query rows per tile (TMEM lanes)
constexpr int kN = 128;  // keys per tile
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;  // S0 [0,128), S1 [128,256), O [256, 256 + D)
constexpr uint64_t kWaitNs = 2000000000ull;

template <int D>
struct TcLayout {
  static constexpr int kHalves = D / 64;         // 64-element (128-byte) column chunks
  static constexpr int kHalf = kM * 128;          // one chunk of a 128-row tile: 16 KB
  static constexpr int kTile = kHalves * kHalf;   // Q, K or V tile
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;           // 2 stages
  static constexpr int kV = kK + 2 * kTile;       // 2 stages
  static constexpr int kP = kV + 2 * kTile;       // 128 rows x 128 keys: 2 chunks
  static constexpr int kBar = kP + 2 * kHalf;
  static constexpr int kBytes = kBar + 128;
  static constexpr int kAlloc = kBytes + 1024;    // slack to align the base to 1 KB
};

enum : int {
  kBarQ = 0,
  kBarK0 = 1,  // K full, stages 0/1
  kBarV0 = 3,  // V full
  kBarE0 = 5,  // stage empty (PV done)
  kBarS0 = 7,  // S buffer full
  kBarP = 9,   // P written by the 128 softmax threads
  kBarO = 10,  // PV done
  kBarDrain = 11,
  kNumBars = 12
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
  using Ly = TcLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (base - raw);

  const int h = blockIdx.x;
  const int s = a.num_decode + static_cast<int>(blockIdx.y);
  const int g = a.group;
  const int hk = h / g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int t0 = __ldg(a.qsl + s);
  const int qn = __ldg(a.qsl + s + 1) - t0;
  const int L = __ldg(a.seq_lens + s);
  if (qn <= 0) return;
  if (L < qn || L > (a.max_blocks << a.bs_log2) || qn > a.max_query_len || L > a.max_seq_len ||
      t0 < 0 || t0 + qn > a.num_tokens) {
    if (blockIdx.x == 0 && blockIdx.z == 0 && threadIdx.x == 0) flag_error(a.err, PA_DEV_BAD_LEN);
    return;
  }
  const int ntiles = (qn + kM - 1) / kM;
  const int tile = ntiles - 1 - static_cast<int>(blockIdx.z);
  if (tile < 0) return;
  const int c = L - qn;
  const int i0 = tile * kM;
  const int i_hi = min(qn, i0 + kM) - 1;
  const int kv_end = c + i_hi + 1;  // keys [0, kv_end) are visible to some row
  const int n = (kv_end + kN - 1) / kN;

  const uint32_t bar0 = base + Ly::kBar;
  const uint32_t tmem_slot = bar0 + 8 * kNumBars;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(sgen + Ly::kBar + 8 * kNumBars + 4);
#define BAR(i) (bar0 + 8u * static_cast<uint32_t>(i))

  if (warp == 5) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(BAR(i), i == kBarP ? 128u : 1u);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (threadIdx.x == 128) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sgen + Ly::kBar + 8 * kNumBars);

  auto give_up = [&]() {
    *abort_flag = 1u;
    flag_error(a.err, PA_DEV_TIMEOUT);
  };

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int32_t* bt = a.block_tables + static_cast<int64_t>(s) * a.max_blocks;
      const int bs = 1 << a.bs_log2;
      const int R = bs < 128 ? bs : 128;  // cache rows per TMA box
      mbar_expect_tx(BAR(kBarQ), Ly::kTile);
#pragma unroll
      for (int hf = 0; hf < Ly::kHalves; ++hf)
        tma_load_2d(base + Ly::kQ + hf * Ly::kHalf, &tm_q, h * D + hf * 64, t0 + i0, BAR(kBarQ));
      int issued_last = -1;
      for (int j = 0; j < n; ++j) {
        const int st = j & 1;
        if (*abort_flag) break;
        if (j >= 2 && !mbar_wait(BAR(kBarE0 + st), ((j >> 1) - 1) & 1, kWaitNs)) {
          give_up();
          break;
        }
        const int p0 = j * kN;
        const int p1 = min(kv_end, p0 + kN);
        const int nbox = (p1 - p0 + R - 1) / R;
        int slots[kN / 8];
        int nvalid = 0;
        for (int b = 0; b < nbox; ++b) {
          const int pos = p0 + b * R;
          const int pb = __ldg(bt + (pos >> a.bs_log2));
          if (pb >= 0 && pb < a.num_blocks) {
            slots[b] = (pb << a.bs_log2) + (pos & (bs - 1));
            ++nvalid;
          } else {
            slots[b] = -1;
            flag_error(a.err, PA_DEV_BAD_BLOCK);
          }
        }
        const uint32_t bytes = static_cast<uint32_t>(nvalid * R * 128 * Ly::kHalves);
        const uint32_t kdst = base + Ly::kK + st * Ly::kTile;
        const uint32_t vdst = base + Ly::kV + st * Ly::kTile;
        mbar_expect_tx(BAR(kBarK0 + st), bytes);
        for (int b = 0; b < nbox; ++b) {
          if (slots[b] < 0) continue;
#pragma unroll
          for (int hf = 0; hf < Ly::kHalves; ++hf)
            tma_load_3d(kdst + hf * Ly::kHalf + b * R * 128, &tm_k, hf * 64, hk, slots[b],
                        BAR(kBarK0 + st));
        }
        mbar_expect_tx(BAR(kBarV0 + st), bytes);
        for (int b = 0; b < nbox; ++b) {
          if (slots[b] < 0) continue;
#pragma unroll
          for (int hf = 0; hf < Ly::kHalves; ++hf)
            tma_load_3d(vdst + hf * Ly::kHalf + b * R * 128, &tm_v, hf * 64, hk, slots[b],
                        BAR(kBarV0 + st));
        }
        issued_last = j;
      }
      // drain: the last (up to) two tiles' copies must have landed before exit
      for (int j = max(0, issued_last - 1); j <= issued_last; ++j) {
        mbar_wait(BAR(kBarK0 + (j & 1)), (j >> 1) & 1, kWaitNs);
        mbar_wait(BAR(kBarV0 + (j & 1)), (j >> 1) & 1, kWaitNs);
      }
      {
        // the Q copy too
        mbar_wait(BAR(kBarQ), 0, kWaitNs);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_bf16(kM, kN, false);
    constexpr uint32_t kIdO = idesc_bf16(kM, D, true);
    const uint32_t tO = tmem + 256;
    auto issue_s = [&](int j) {
      const int st = j & 1;
      const uint32_t q0 = base + Ly::kQ, k0 = base + Ly::kK + st * Ly::kTile;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * Ly::kHalf + (kk & 3) * 32;
        mma_f16_ss(tmem + st * 128, smem_desc_sw128(q0 + off, 16, 1024),
                   smem_desc_sw128(k0 + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
      }
      mma_commit(BAR(kBarS0 + st));
    };
    bool ok = mbar_wait(BAR(kBarQ), 0, kWaitNs) && mbar_wait(BAR(kBarK0), 0, kWaitNs);
    if (!ok) give_up();
    tc_fence_after();
    if (ok && lane == 0) issue_s(0);
    __syncwarp();
    for (int j = 0; ok && j < n; ++j) {
      const int st = j & 1;
      if (j + 1 < n) {
        ok = !*abort_flag && mbar_wait(BAR(kBarK0 + ((j + 1) & 1)), ((j + 1) >> 1) & 1, kWaitNs);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) issue_s(j + 1);
        __syncwarp();
      }
      ok = !*abort_flag && mbar_wait(BAR(kBarP), j & 1, kWaitNs) &&
           mbar_wait(BAR(kBarV0 + st), (j >> 1) & 1, kWaitNs);
      if (!ok) break;
      tc_fence_after();
      const int live = kv_end - j * kN;  // rows [live, 128) of this V tile are not keys
      if (live < kN) {
        uint8_t* vt = sgen + Ly::kV + st * Ly::kTile;
        const int nbytes = (kN - live) * 128;
        for (int hf = 0; hf < Ly::kHalves; ++hf) {
          uint4* p = reinterpret_cast<uint4*>(vt + hf * Ly::kHalf + live * 128);
          for (int x = lane; x < nbytes / 16; x += 32) p[x] = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) {
        const uint32_t p0 = base + Ly::kP, v0 = base + Ly::kV + st * Ly::kTile;
#pragma unroll
        for (int kk = 0; kk < kN / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * Ly::kHalf + (kk & 3) * 32;
          mma_f16_ss(tO, smem_desc_sw128(p0 + aoff, 16, 1024),
                     smem_desc_sw128(v0 + kk * 2048, Ly::kHalf, 1024), kIdO,
                     (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(BAR(kBarO));
        mma_commit(BAR(kBarE0 + st));
      }
      __syncwarp();
    }
    if (!ok) give_up();
    // drain: every MMA this thread issued has completed once this arrives
    if (lane == 0) mma_commit(BAR(kBarDrain));
    __syncwarp();
    mbar_wait(BAR(kBarDrain), 0, kWaitNs);
  } else {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;  // 0..127
    const int i = i0 + r;
    const bool row_ok = i < qn;
    const int lim = c + i;  // last key position this row sees
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t prow = base + Ly::kP + r * 128;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      ok = !*abort_flag && mbar_wait(BAR(kBarS0 + (j & 1)), (j >> 1) & 1, kWaitNs);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(tmem + lane_off + (j & 1) * 128 + cc * 32, sr[cc]);
      tmem_wait_ld();
      const int key0 = j * kN;
      const bool full = key0 + kN - 1 <= lim && key0 + kN <= kv_end;
      float mt = -INFINITY;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float v = __uint_as_float(sr[cc][e]) * a.scale_log2;
          const int pos = key0 + cc * 32 + e;
          if (!full && (pos > lim || pos >= kv_end)) v = -INFINITY;
          sr[cc][e] = __float_as_uint(v);
          mt = fmaxf(mt, v);
        }
      const float m_new = mt > m_used + 8.f ? mt : m_used;
      const float ref = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = m_used == -INFINITY ? 0.f : ex2(m_used - ref);
      float rs = 0.f;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float p = ex2(__uint_as_float(sr[cc][e]) - ref);
          rs += p;
          sr[cc][e] = __float_as_uint(p);
        }
      l = l * alpha + rs;
      if (j > 0) {
        ok = !*abort_flag && mbar_wait(BAR(kBarO), (j - 1) & 1, kWaitNs);
        if (!ok) break;
        tc_fence_after();
      }
      const bool need = j > 0 && m_new != m_used;
      if (__any_sync(0xffffffffu, need)) {
        const float f = need ? alpha : 1.f;
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + 256 + cc * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
          tmem_st32(tmem + lane_off + 256 + cc * 32, o);
        }
        tmem_wait_st();
      }
      m_used = m_new;
      // P row -> smem, K-major with the 128-byte swizzle: 16-byte chunk q of
      // row r in a 64-key half lands at chunk q ^ (r & 7).
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          const int k = hf * 64 + q8 * 8;
          const uint32_t* v = &sr[k >> 5][k & 31];
          uint4 w;
          w.x = pack_bf16(__uint_as_float(v[0]), __uint_as_float(v[1]));
          w.y = pack_bf16(__uint_as_float(v[2]), __uint_as_float(v[3]));
          w.z = pack_bf16(__uint_as_float(v[4]), __uint_as_float(v[5]));
          w.w = pack_bf16(__uint_as_float(v[6]), __uint_as_float(v[7]));
          const uint32_t addr = prow + hf * Ly::kHalf + ((q8 ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(w.x),
                       "r"(w.y), "r"(w.z), "r"(w.w)
                       : "memory");
        }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(BAR(kBarP));
    }
    if (ok) ok = !*abort_flag && mbar_wait(BAR(kBarO), (n - 1) & 1, kWaitNs);
    if (!ok) {
      give_up();
    } else {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                            static_cast<int64_t>(t0 + (row_ok ? i : 0)) * a.out_stride +
                            static_cast<int64_t>(h) * D;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + 256 + cc * 32, o);
        tmem_wait_ld();
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(o[q4 * 8 + 0]) * inv, __uint_as_float(o[q4 * 8 + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(o[q4 * 8 + 2]) * inv, __uint_as_float(o[q4 * 8 + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(o[q4 * 8 + 4]) * inv, __uint_as_float(o[q4 * 8 + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(o[q4 * 8 + 6]) * inv, __uint_as_float(o[q4 * 8 + 7]) * inv);
            dst[q4] = w;
          }
        }
      }
    }
  }
#undef BAR
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
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

bool encode_q(CUtensorMap* m, const AttnArgs& a) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.hq) * a.head_dim,
                              static_cast<cuuint64_t>(a.num_tokens)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.q_stride) * 2};
  const cuuint32_t box[2] = {64, kM};
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

template <int D>
cudaError_t launch_tc_d(const AttnArgs& a, cudaStream_t st) {
  using Ly = TcLayout<D>;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::kAlloc);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  CUtensorMap mq, mk, mv;
  if (!encode_q(&mq, a) || !encode_cache(&mk, a.k_cache, a) || !encode_cache(&mv, a.v_cache, a))
    return cudaErrorNotSupported;  // nothing launched: the caller takes the general kernel
  dim3 grid(a.hq, a.num_seqs - a.num_decode, (a.max_query_len + kM - 1) / kM);
  count_launch();
  prefill_tc_kernel<D><<<grid, kThreads, Ly::kAlloc, st>>>(mq, mk, mv, a);
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(const AttnArgs& a) {
  const char* env = getenv("PA_PREFILL_IMPL");
  if (env && strcmp(env, "mma") == 0) return false;
  if (a.head_dim != 64 && a.head_dim != 128) return false;
  if (a.bs_log2 < 3) return false;  // TMA boxes of >= 8 rows keep 1 KB swizzle alignment
  if ((a.q_stride * 2) % 16 != 0) return false;
  if ((reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.k_cache) |
       reinterpret_cast<uintptr_t>(a.v_cache)) & 15u)
    return false;
  if ((a.max_query_len + kM - 1) / kM > 65535) return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const AttnArgs& a, cudaStream_t st) {
  if (a.num_seqs - a.num_decode <= 0 || a.max_query_len <= 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_tc_d<128>(a, st) : launch_tc_d<64>(a, st);
}

}  // namespace pa
