// Router: logits with fused bias, then per-token top-k (warp shuffles),
// sigmoid and renormalisation of the selected scores.
//
// "Add GLM-5.3-Flash (glm5next) support with ROCmFP mix qtypes (105/106)",
// section "MoE FFN (REAL routed expert execution)": the router computes
// sigmoid(moe_gate @ input + moe_exp_probs_b), takes the top 8 experts and
// normalises their weights.  Ties go to the lower expert index (deterministic
// top-k, "feat(glm53): add device-resident HIP backend for MI350P", "Key
// changes").
#include <cuda_bf16.h>

#include "moe_kernels.h"
#include "ptx.cuh"
#include "route_common.cuh"

namespace moe {
namespace {

constexpr int kRouterWarps = 4;    // experts per CTA (one per warp)
constexpr int kRouterTokTile = 8;  // tokens per CTA
constexpr int kLoadBatch = 8;      // 16-byte router loads in flight per lane

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// grid (ceil(E / 4), ceil(T / 8)), 128 threads.  The CTA stages its 8 token
// rows in shared memory; each warp streams one router row, issuing 8 16-byte
// loads per lane before using any of them, and keeps 8 fp32 partial sums,
// reduced across the warp at the end.
__global__ void __launch_bounds__(128) router_logits_simt_kernel(const uint16_t* __restrict__ x,
                                                                 const uint16_t* __restrict__ wr,
                                                                 const float* __restrict__ b,
                                                                 float* __restrict__ z, int T,
                                                                 int H, int E) {
  extern __shared__ uint4 xs[];  // [kRouterTokTile][H / 8]
  pdl_wait();
  const int chunks = H / 8;
  const int t0 = blockIdx.y * kRouterTokTile;
  const int nt = min(kRouterTokTile, T - t0);
  const uint4* xg = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t0) * H);
  for (int i = threadIdx.x; i < nt * chunks; i += blockDim.x) xs[i] = __ldg(xg + i);
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouterWarps + warp;
  if (e < E) {
    float acc[kRouterTokTile];
#pragma unroll
    for (int t = 0; t < kRouterTokTile; ++t) acc[t] = 0.f;
    const uint4* wrow = reinterpret_cast<const uint4*>(wr + static_cast<size_t>(e) * H);
    for (int c0 = lane; c0 < chunks; c0 += 32 * kLoadBatch) {
      uint4 wv[kLoadBatch];
#pragma unroll
      for (int i = 0; i < kLoadBatch; ++i) {
        const int c = c0 + 32 * i;
        wv[i] = c < chunks ? __ldg(wrow + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < kLoadBatch; ++i) {
        const int c = c0 + 32 * i;
        if (c < chunks) {
          float wf[8];
          bf16x8_to_f32(wv[i], wf);
#pragma unroll
          for (int t = 0; t < kRouterTokTile; ++t) {
            if (t < nt) {
              float xf[8];
              bf16x8_to_f32(xs[t * chunks + c], xf);
#pragma unroll
              for (int j = 0; j < 8; ++j) acc[t] = fmaf(xf[j], wf[j], acc[t]);
            }
          }
        }
      }
    }
    const float bias = b[e];
#pragma unroll
    for (int t = 0; t < kRouterTokTile; ++t) {
      float v = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && t < nt) z[static_cast<size_t>(t0 + t) * E + e] = v + bias;
    }
  }
  pdl_launch_dependents();
}

// One warp per token: top-k, sigmoid, renormalisation.
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ z, int T, int E,
                                                   int k, int32_t* __restrict__ idx,
                                                   float* __restrict__ w) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t < T) {
    int e;
    float wv;
    warp_topk(z + static_cast<size_t>(t) * E, E, k, &e, &wv);
    if (lane < k) {
      idx[static_cast<size_t>(t) * k + lane] = e;
      w[static_cast<size_t>(t) * k + lane] = wv;
    }
  }
  pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_router_logits_simt(const uint16_t* x, const uint16_t* w_router, const float* b,
                                      float* z, int T, int H, int E, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(kRouterTokTile) * H * 2;
  cudaError_t err = cudaFuncSetAttribute(router_logits_simt_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const dim3 grid((E + kRouterWarps - 1) / kRouterWarps, (T + kRouterTokTile - 1) / kRouterTokTile);
  return launch_pdl(router_logits_simt_kernel, grid, dim3(32 * kRouterWarps), smem, s, x,
                    w_router, b, z, T, H, E);
}

cudaError_t launch_topk(const float* z, int T, int E, int k, int32_t* idx, float* w,
                        cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(topk_kernel, dim3((T + 7) / 8), dim3(256), 0, s, z, T, E, k, idx, w);
}

}  // namespace moe
