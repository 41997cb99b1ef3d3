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

namespace moe {
namespace {

constexpr int kRouterWarps = 8;    // experts per CTA (one per warp)
constexpr int kRouterTokTile = 8;  // tokens per CTA

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// grid (ceil(E / 8), ceil(T / 8)), 256 threads.  The CTA stages its 8 token
// rows in shared memory; each warp streams one router row with 16-byte loads
// and keeps 8 fp32 partial sums, reduced across the warp at the end.
__global__ void __launch_bounds__(256) router_logits_simt_kernel(const uint16_t* __restrict__ x,
                                                                 const uint16_t* __restrict__ wr,
                                                                 const float* __restrict__ b,
                                                                 float* __restrict__ z, int T,
                                                                 int H, int E) {
  extern __shared__ uint4 xs[];  // [kRouterTokTile][H / 8]
  const int chunks = H / 8;
  const int t0 = blockIdx.y * kRouterTokTile;
  const int nt = min(kRouterTokTile, T - t0);
  const uint4* xg = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t0) * H);
  for (int i = threadIdx.x; i < nt * chunks; i += blockDim.x) xs[i] = __ldg(xg + i);
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouterWarps + warp;
  if (e >= E) return;
  float acc[kRouterTokTile];
#pragma unroll
  for (int t = 0; t < kRouterTokTile; ++t) acc[t] = 0.f;
  const uint4* wrow = reinterpret_cast<const uint4*>(wr + static_cast<size_t>(e) * H);
  for (int c = lane; c < chunks; c += 32) {
    float wf[8];
    bf16x8_to_f32(__ldg(wrow + c), wf);
#pragma unroll
    for (int t = 0; t < kRouterTokTile; ++t) {
      if (t < nt) {
        float xf[8];
        bf16x8_to_f32(xs[t * chunks + c], xf);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[t] = fmaf(xf[i], wf[i], acc[t]);
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

// Order-preserving map of a float onto uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t float_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

constexpr int kVPL = kMaxE / 32;  // values per lane

// One warp per token.  Lane L holds experts L, L+32, ...; each of the k rounds
// takes the warp-wide maximum of the 64-bit key (score key << 32 | ~e), so the
// larger score wins and an exact tie goes to the lower expert index.  Slot j
// ends in lane j, which applies the sigmoid; the warp sums the k scores and
// each slot is divided by the sum.
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ z, int T, int E,
                                                   int k, int32_t* __restrict__ idx,
                                                   float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* zr = z + static_cast<size_t>(t) * E;
  uint32_t keys[kVPL];
#pragma unroll
  for (int i = 0; i < kVPL; ++i) {
    const int e = i * 32 + lane;
    keys[i] = e < E ? float_key(__ldg(zr + e)) : 0u;
  }
  uint32_t taken = 0;
  int my_e = 0;
  float my_z = 0.f;
  for (int j = 0; j < k; ++j) {
    uint64_t best = 0;
#pragma unroll
    for (int i = 0; i < kVPL; ++i) {
      const int e = i * 32 + lane;
      if (e < E && !((taken >> i) & 1u)) {
        const uint64_t key = (static_cast<uint64_t>(keys[i]) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(e));
        best = key > best ? key : best;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint64_t other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    const int e_win = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(best & 0xFFFFFFFFu));
    if ((e_win & 31) == lane) taken |= 1u << (e_win >> 5);
    if (lane == j) {
      my_e = e_win;
      my_z = key_float(static_cast<uint32_t>(best >> 32));
    }
  }
  const float s = lane < k ? 1.0f / (1.0f + expf(-my_z)) : 0.f;
  float sum = s;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    idx[static_cast<size_t>(t) * k + lane] = my_e;
    w[static_cast<size_t>(t) * k + lane] = s / sum;
  }
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
  dim3 grid((E + kRouterWarps - 1) / kRouterWarps, (T + kRouterTokTile - 1) / kRouterTokTile);
  router_logits_simt_kernel<<<grid, 256, smem, s>>>(x, w_router, b, z, T, H, E);
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* z, int T, int E, int k, int32_t* idx, float* w,
                        cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  topk_kernel<<<(T + 7) / 8, 256, 0, s>>>(z, T, E, k, idx, w);
  return cudaGetLastError();
}

}  // namespace moe
