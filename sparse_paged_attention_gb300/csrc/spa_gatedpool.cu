// spa_gatedpool.cu - the KV compressor's gated pool: R buffered rows fold into one compressed
// entry, each channel weighted by a softmax of its gates over the R rows (FreeToken PR 633, call
// paths and "Changes": the compressor's decode step, a maximum over R then a weighted pass).
//
//   out[b, d] = sum_r e^(g[b,r,d] - M) kv[b,r,d] / sum_r e^(g[b,r,d] - M),   M = max_r g[b,r,d]
//
// The work is a pure stream of 8·R·D bytes per entry with no reuse, so HBM (and, at the small
// shapes the decode step runs, launch latency) bounds it.  One CTA takes 32·VEC channels of one
// entry; its nw = ceil(R / 8) warps (at most 16) split the R rows, row r going to warp r mod nw, so
// that a warp holds about eight rows.  Each lane keeps an online maximum, denominator and weighted
// sum for VEC adjacent channels over a one-pass read (no second read of the rows for the maximum),
// loading a batch of eight rows (16 loads) before any arithmetic.  With one warp the lane writes
// its channels directly; otherwise the warps' states meet in shared memory and 16 lanes per channel
// merge them by the same rescaling rule in a shuffle tree.
#include <cuda_bf16.h>

#include "spa_launch.h"

namespace spa {

namespace {

constexpr int kRowsPerBatch = 8;

// Rescale-and-add of one partial state (m2, l2, a2) into (m, l, a); -inf maxima stand for "no
// row yet" (their l and a are 0).
__device__ __forceinline__ void merge_state(float& m, float& l, float& a, float m2, float l2,
                                            float a2) {
  const float mn = fmaxf(m, m2);
  const float ref = mn == -INFINITY ? 0.f : mn;
  const float c1 = expf(m - ref), c2 = expf(m2 - ref);
  l = l * c1 + l2 * c2;
  a = a * c1 + a2 * c2;
  m = mn;
}

__device__ __forceinline__ void store_out(const GatedPoolArgs& g, long long b, int d, float o) {
  if (g.out_bf16)
    reinterpret_cast<__nv_bfloat16*>(g.out)[b * g.out_sb + d] = __float2bfloat16_rn(o);
  else
    reinterpret_cast<float*>(g.out)[b * g.out_sb + d] = o;
}

template <int VEC>
__global__ void __launch_bounds__(kGatedPoolMaxWarps * 32)
    gated_pool_kernel(const GatedPoolArgs g) {
  constexpr int CH = 32 * VEC;  // channels per CTA
  __shared__ float s_m[kGatedPoolMaxWarps][CH], s_l[kGatedPoolMaxWarps][CH],
      s_a[kGatedPoolMaxWarps][CH];
  const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunks = (g.D + CH - 1) / CH;
  const long long b = blockIdx.x / chunks;
  const int c0 = (int)(blockIdx.x % chunks) * CH;
  const int d = c0 + lane * VEC;
  const bool live = d < g.D;  // the vector path needs D % VEC == 0, so d + VEC - 1 < D too
  pdl_launch_dependents();
  pdl_wait();   // nothing global before the grid before this one is done

  float m[VEC], l[VEC], acc[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) m[v] = -INFINITY, l[v] = 0.f, acc[v] = 0.f;

  const float* kvb = g.kv + b * g.kv_sb + d;
  const float* gb = g.gate + b * g.gate_sb + d;
  for (int r0 = warp; r0 < g.R; r0 += nw * kRowsPerBatch) {
    float x[kRowsPerBatch][VEC], s[kRowsPerBatch][VEC];
#pragma unroll
    for (int u = 0; u < kRowsPerBatch; ++u) {
      const int r = r0 + u * nw;
      if (live && r < g.R) {
        if constexpr (VEC == 4) {
          const float4 xv = __ldg(reinterpret_cast<const float4*>(kvb + (long long)r * g.kv_sr));
          const float4 sv = __ldg(reinterpret_cast<const float4*>(gb + (long long)r * g.gate_sr));
          x[u][0] = xv.x, x[u][1] = xv.y, x[u][2] = xv.z, x[u][3] = xv.w;
          s[u][0] = sv.x, s[u][1] = sv.y, s[u][2] = sv.z, s[u][3] = sv.w;
        } else {
          x[u][0] = __ldg(kvb + (long long)r * g.kv_sr);
          s[u][0] = __ldg(gb + (long long)r * g.gate_sr);
        }
      } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) x[u][v] = 0.f, s[u][v] = -INFINITY;
      }
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      float mb = s[0][v];
#pragma unroll
      for (int u = 1; u < kRowsPerBatch; ++u) mb = fmaxf(mb, s[u][v]);
      const float mn = fmaxf(m[v], mb);
      const float ref = mn == -INFINITY ? 0.f : mn;
      const float c = expf(m[v] - ref);
      float lv = l[v] * c, av = acc[v] * c;
#pragma unroll
      for (int u = 0; u < kRowsPerBatch; ++u) {
        const float e = expf(s[u][v] - ref);
        lv += e;
        av = fmaf(e, x[u][v], av);
      }
      m[v] = mn, l[v] = lv, acc[v] = av;
    }
  }

  if (nw == 1) {  // this lane saw every row of its channels
    if (live) {
#pragma unroll
      for (int v = 0; v < VEC; ++v) store_out(g, b, d + v, g.R == 0 ? 0.f : acc[v] / l[v]);
    }
    return;
  }
#pragma unroll
  for (int v = 0; v < VEC; ++v) {
    s_m[warp][lane * VEC + v] = m[v];
    s_l[warp][lane * VEC + v] = l[v];
    s_a[warp][lane * VEC + v] = acc[v];
  }
  __syncthreads();
  // lanes 0-15 of a warp merge one channel, lanes 16-31 the next; lane (tid & 15) brings the state
  // of warp (tid & 15).  CH and the stride 2·nw are even, so both halves of a warp run the same
  // trips and the full-mask shuffles are warp-uniform.
  const int sub = threadIdx.x & 15;
  for (int c = threadIdx.x >> 4; c < CH; c += blockDim.x >> 4) {
    float mm = -INFINITY, ll = 0.f, aa = 0.f;
    if (sub < nw) mm = s_m[sub][c], ll = s_l[sub][c], aa = s_a[sub][c];
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, mm, o);
      const float l2 = __shfl_xor_sync(0xffffffffu, ll, o);
      const float a2 = __shfl_xor_sync(0xffffffffu, aa, o);
      merge_state(mm, ll, aa, m2, l2, a2);
    }
    if (sub == 0 && c0 + c < g.D) store_out(g, b, c0 + c, aa / ll);
  }
}

}  // namespace

cudaError_t launch_gated_pool(const GatedPoolArgs& g, int num_sms, cudaStream_t stream) {
  if (g.B == 0 || g.D == 0) return cudaSuccess;
  // 16-byte loads only when they still leave a CTA for every SM: at the decode step's sizes the
  // narrower CTAs spread the rows over more SMs, which matters more than the load width
  int vec = gated_pool_vector_width(g);
  if (vec == 4 && (long long)g.B * ((g.D + 127) / 128) < num_sms) vec = 1;
  const long long chunks = (g.D + 32LL * vec - 1) / (32LL * vec);
  const long long blocks = (long long)g.B * chunks;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  int nw = (g.R + kRowsPerBatch - 1) / kRowsPerBatch;  // about one batch of rows per warp
  nw = nw < 1 ? 1 : (nw > kGatedPoolMaxWarps ? kGatedPoolMaxWarps : nw);
  const bool pdl = 2 * blocks <= num_sms;
  if (vec == 4)
    return launch_with_pdl(gated_pool_kernel<4>, dim3((unsigned)blocks), dim3(nw * 32), 0, stream,
                           pdl, g);
  return launch_with_pdl(gated_pool_kernel<1>, dim3((unsigned)blocks), dim3(nw * 32), 0, stream,
                         pdl, g);
}

}  // namespace spa
