// KV-cache scatter through slot_mapping and copy-on-write block copies.
//
// Both are pure data movement: 16-byte vector loads and stores, consecutive
// threads on consecutive 16-byte pieces of one token row (or one block), so
// every warp moves 512 contiguous bytes per instruction.
#include "common.cuh"
#include "internal.h"

namespace pa {

// One thread per 16-byte piece of a [num_kv_heads * head_dim] token row.
// "vLLM Continuous Batching：从 Forward Shape 理解两个核心参数" §2.3补充 第一步:
// token t's K/V go to slot_mapping[t] = block * block_size + offset, which is
// row `slot` of the cache viewed as [num_blocks * block_size, kv_heads, dim].
__global__ void __launch_bounds__(256) write_kv_kernel(const uint4* __restrict__ k,
                                                       const uint4* __restrict__ v, int64_t ks,
                                                       int64_t vs, uint4* __restrict__ kc,
                                                       uint4* __restrict__ vc,
                                                       const int32_t* __restrict__ slots, int T,
                                                       int vec_per_row, int64_t num_slots,
                                                       uint32_t* err) {
  // One warp per token row (grid-stride over tokens), the lanes across the
  // row's 16-byte pieces: no index division, and each lane's loads of a row
  // are issued before its stores.
  const int lane = threadIdx.x & 31;
  const int nwarps = static_cast<int>((gridDim.x * blockDim.x) >> 5);
  for (int t = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5); t < T;
       t += nwarps) {
    const int slot = __ldg(slots + t);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (lane == 0) flag_error(err, PA_DEV_BAD_SLOT);
      continue;
    }
    const uint4* kr = k + static_cast<int64_t>(t) * ks;
    const uint4* vr = v + static_cast<int64_t>(t) * vs;
    uint4* kd = kc + static_cast<int64_t>(slot) * vec_per_row;
    uint4* vd = vc + static_cast<int64_t>(slot) * vec_per_row;
    int c = lane;
    for (; c + 96 < vec_per_row; c += 128) {
      uint4 a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        a[u] = __ldg(kr + c + 32 * u);
        b[u] = __ldg(vr + c + 32 * u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        kd[c + 32 * u] = a[u];
        vd[c + 32 * u] = b[u];
      }
    }
    for (; c < vec_per_row; c += 32) {
      const uint4 a = __ldg(kr + c);
      const uint4 b = __ldg(vr + c);
      kd[c] = a;
      vd[c] = b;
    }
  }
}

__global__ void __launch_bounds__(256) write_kv_fp8_kernel(const uint4* __restrict__ k,
                                                           const uint4* __restrict__ v, int64_t ks,
                                                           int64_t vs, uint2* __restrict__ kc,
                                                           uint2* __restrict__ vc,
                                                           const int32_t* __restrict__ slots,
                                                           int T, int vec_per_row,
                                                           int64_t num_slots, float inv_k,
                                                           float inv_v, uint32_t* err) {
  const int64_t total = static_cast<int64_t>(T) * vec_per_row;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / vec_per_row);
    const int c = static_cast<int>(i - static_cast<int64_t>(t) * vec_per_row);
    const int slot = __ldg(slots + t);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (c == 0) flag_error(err, PA_DEV_BAD_SLOT);
      continue;
    }
    const int64_t o = static_cast<int64_t>(slot) * vec_per_row + c;
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      const uint4 w = __ldg(kv ? v + t * vs + c : k + t * ks + c);
      const float inv = kv ? inv_v : inv_k;
      const uint32_t in[4] = {w.x, w.y, w.z, w.w};
      uint32_t q[2] = {0u, 0u};
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&in[p]);
        const float2 f = make_float2(__low2float(b) * inv, __high2float(b) * inv);
        const uint32_t two = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
        q[p >> 1] |= two << (16 * (p & 1));
      }
      (kv ? vc : kc)[o] = make_uint2(q[0], q[1]);
    }
  }
}

// blockIdx.y = pair; threads stride over the block's 16-byte pieces.
// "vLLM 原理" §2.1: the fresh block receives the shared block's whole contents.
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4* __restrict__ kc,
                                                          uint4* __restrict__ vc,
                                                          const int32_t* __restrict__ pairs,
                                                          int num_blocks, int vec_per_block,
                                                          uint32_t* err) {
  const int p = blockIdx.y;
  const int src = __ldg(pairs + 2 * p), dst = __ldg(pairs + 2 * p + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(err, PA_DEV_BAD_PAIR);
    return;
  }
  const int64_t so = static_cast<int64_t>(src) * vec_per_block;
  const int64_t d = static_cast<int64_t>(dst) * vec_per_block;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < vec_per_block;
       i += gridDim.x * blockDim.x) {
    const uint4 a = kc[so + i];
    const uint4 b = vc[so + i];
    kc[d + i] = a;
    vc[d + i] = b;
  }
}

// Block moves between two pools (blockIdx.y = pair); either pool may live in
// host memory the device can reach.  Same 16-byte streaming as the block copy.
__global__ void __launch_bounds__(256) swap_blocks_kernel(const uint4* __restrict__ sk,
                                                          const uint4* __restrict__ sv,
                                                          uint4* __restrict__ dk,
                                                          uint4* __restrict__ dv,
                                                          const int32_t* __restrict__ pairs,
                                                          int src_blocks, int dst_blocks,
                                                          int vec_per_block, uint32_t* err) {
  const int p = blockIdx.y;
  const int src = __ldg(pairs + 2 * p), dst = __ldg(pairs + 2 * p + 1);
  if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(err, PA_DEV_BAD_PAIR);
    return;
  }
  const int64_t so = static_cast<int64_t>(src) * vec_per_block;
  const int64_t d = static_cast<int64_t>(dst) * vec_per_block;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < vec_per_block;
       i += gridDim.x * blockDim.x) {
    const uint4 a = sk[so + i];
    const uint4 b = sv[so + i];
    dk[d + i] = a;
    dv[d + i] = b;
  }
}

cudaError_t launch_write_kv(const void* k, const void* v, int64_t ks, int64_t vs, void* kc,
                            void* vc, const int32_t* slots, int T, int num_blocks, int bs,
                            int row_elems, uint32_t* err, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int vpr = row_elems / 8;
  int64_t blocks = (static_cast<int64_t>(T) + 7) / 8;  // a warp per token, 8 warps per block
  if (blocks > 152 * 16) blocks = 152 * 16;
  count_launch();
  write_kv_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), ks / 8, vs / 8,
      static_cast<uint4*>(kc), static_cast<uint4*>(vc), slots, T, vpr,
      static_cast<int64_t>(num_blocks) * bs, err);
  return cudaGetLastError();
}

cudaError_t launch_write_kv_fp8(const void* k, const void* v, int64_t ks, int64_t vs, void* kc,
                                void* vc, const int32_t* slots, int T, int num_blocks, int bs,
                                int row_elems, float inv_k_scale, float inv_v_scale,
                                uint32_t* err, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int vpr = row_elems / 8;
  const int64_t total = static_cast<int64_t>(T) * vpr;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  count_launch();
  write_kv_fp8_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), ks / 8, vs / 8,
      static_cast<uint2*>(kc), static_cast<uint2*>(vc), slots, T, vpr,
      static_cast<int64_t>(num_blocks) * bs, inv_k_scale, inv_v_scale, err);
  return cudaGetLastError();
}

cudaError_t launch_copy_blocks(void* kc, void* vc, const int32_t* pairs, int n, int num_blocks,
                               int block_elems, uint32_t* err, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int vpb = block_elems / 8;
  int bx = (vpb + 255) / 256;
  if (bx > 8) bx = 8;
  count_launch();
  copy_blocks_kernel<<<dim3(bx, n), 256, 0, st>>>(static_cast<uint4*>(kc), static_cast<uint4*>(vc),
                                                   pairs, num_blocks, vpb, err);
  return cudaGetLastError();
}

cudaError_t launch_swap_blocks(const void* sk, const void* sv, void* dk, void* dv,
                               const int32_t* pairs, int n, int src_blocks, int dst_blocks,
                               int block_elems, uint32_t* err, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int vpb = block_elems / 8;
  int bx = (vpb + 255) / 256;
  if (bx > 8) bx = 8;
  count_launch();
  swap_blocks_kernel<<<dim3(bx, n), 256, 0, st>>>(
      static_cast<const uint4*>(sk), static_cast<const uint4*>(sv), static_cast<uint4*>(dk),
      static_cast<uint4*>(dv), pairs, src_blocks, dst_blocks, vpb, err);
  return cudaGetLastError();
}

}  // namespace pa
