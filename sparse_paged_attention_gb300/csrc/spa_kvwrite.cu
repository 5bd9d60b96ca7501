// spa_kvwrite.cu - paged KV write: the rows of new tokens go to their pool slots, copied (bf16
// pools) or quantised to e4m3 with one scale per token and kv_head (FreeToken clone PR 3, "Perf/kv
// fp8 read path": the per-(token, kv_head) K and V scales its read path folds back in).
//
// bf16 pools: one warp per (token, K or V) row, copied in 16-byte chunks.  e4m3 pools: one warp per
// token.  A row of D bf16 values is D / 8 16-byte chunks, at most two per lane (D <= 512): the warp
// issues the loads of both rows (four chunks a lane) before any arithmetic, reduces each row's
// max|x| with shuffles, and writes each row's codes (8 bytes per chunk) and scale.  The kernel is bound by HBM: per token it reads 4·D
// bytes and writes 2·D (e4m3) or 4·D (bf16) bytes plus the scales.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "spa_launch.h"

namespace spa {

namespace {

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// |x| of the eight bf16 values of a 16-byte chunk, maximum
__device__ __forceinline__ float chunk_absmax(const uint4& u) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, fabsf(bf16_bits_to_f32(w[i] & 0xFFFFu)));
    m = fmaxf(m, fabsf(bf16_bits_to_f32(w[i] >> 16)));
  }
  return m;
}

// eight bf16 values / scale (IEEE fp32 division) -> eight e4m3 codes (round to nearest even,
// saturating), first value in the lowest byte
__device__ __forceinline__ uint2 chunk_to_e4m3(const uint4& u, float scale) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = __fdiv_rn(bf16_bits_to_f32(w[i] & 0xFFFFu), scale);
    const float b = __fdiv_rn(bf16_bits_to_f32(w[i] >> 16), scale);
    c[i] = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

template <bool kFp8>
__global__ void __launch_bounds__(256) kv_write_kernel(const KvWriteArgs a) {
  const long long warp_id = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp_id >= (kFp8 ? 1LL : 2LL) * a.T) return;  // (warp-uniform)
  const int t = kFp8 ? (int)warp_id : (int)(warp_id >> 1), kv = kFp8 ? 0 : (int)(warp_id & 1);

  // the slot of the token's position in its sequence's pages
  const int x = __ldg(a.positions + t);
  const int b = a.seq_of_token ? __ldg(a.seq_of_token + t) : 0;
  long long row = -1;
  if (x >= 0 && b >= 0 && b < a.B) {
    const int page = x / a.ps;
    if (page < a.bt_stride) {
      const int blk = __ldg(a.bt + (size_t)b * a.bt_stride + page);
      if (blk >= 0 && (long long)blk < a.num_blocks) row = (long long)blk * a.ps + x % a.ps;
    }
  }
  if (row < 0) {
    if (lane == 0 && kv == 0) flag_error(SPA_ERR_INDEX);
    return;
  }

  const uint4* src = reinterpret_cast<const uint4*>((kv ? a.v : a.k) + (size_t)t * a.D * 2);
  const int nch = a.D >> 3;  // 16-byte chunks of eight bf16 values
  if (!kFp8) {
    uint4* dst = reinterpret_cast<uint4*>(a.kv + ((size_t)row * 2 + kv) * a.D * 2);
    for (int c = lane; c < nch; c += 32) dst[c] = __ldg(src + c);
    return;
  }
  const uint4* srcv = reinterpret_cast<const uint4*>(a.v + (size_t)t * a.D * 2);
  uint4 u[2], w[2];
  float amax = 0.f, vmax = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int c = lane + 32 * i;
    u[i] = c < nch ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
    w[i] = c < nch ? __ldg(srcv + c) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    amax = fmaxf(amax, chunk_absmax(u[i]));
    vmax = fmaxf(vmax, chunk_absmax(w[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
  }
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  const float vscale = vmax > 0.f ? __fdiv_rn(vmax, 448.f) : 1.f;
  uint2* dst = reinterpret_cast<uint2*>(a.kv + ((size_t)row * 2) * a.D);
  uint2* dstv = reinterpret_cast<uint2*>(a.kv + ((size_t)row * 2 + 1) * a.D);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int c = lane + 32 * i;
    if (c < nch) {
      dst[c] = chunk_to_e4m3(u[i], scale);
      dstv[c] = chunk_to_e4m3(w[i], vscale);
    }
  }
  if (lane == 0) {
    a.k_scale[row] = scale;
    a.v_scale[row] = vscale;
  }
}

}  // namespace

// This translation unit's copy of the device error word (see spa_device.cuh).
cudaError_t read_and_clear_kv_write_error_word(int* value) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_spa_error, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_spa_error, &zero, sizeof(int));
}

cudaError_t launch_kv_write(const KvWriteArgs& a, bool fp8, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  const long long threads = (fp8 ? 1LL : 2LL) * a.T * 32;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  if (fp8)
    kv_write_kernel<true><<<blocks, 256, 0, stream>>>(a);
  else
    kv_write_kernel<false><<<blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace spa
