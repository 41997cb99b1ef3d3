// Fixed-order weighted combination of per-row expert outputs:
//   out[t] = sum_{j} w[t][j] * y_perm[row_of[t][j]] + y_perm[k*T + t]
// ("Weighted combination of expert outputs" with the shared expert, "Add
// GLM-5.3-Flash (glm5next) support with ROCmFP mix qtypes (105/106)",
// section "What Executes vs. TODO", item 3).  Every output element is summed
// by one thread in slot order, so the result is the same bits on every run.
// With `accumulate`, the sum starts from out's entry value (a residual).
#include "moe_kernels.h"
#include "ptx.cuh"
#include "route_common.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y,
                                                      const int32_t* __restrict__ row_of,
                                                      const float* __restrict__ w, int T, int H,
                                                      int k, bool accumulate,
                                                      float* __restrict__ out) {
  __shared__ int rows[kMaxTopK + 1];
  __shared__ float wt[kMaxTopK];
  pdl_wait();
  pdl_launch_dependents();  // dependents wait for this grid's completion themselves
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < k) {
      rows[threadIdx.x] = row_of[static_cast<size_t>(t) * k + threadIdx.x];
      wt[threadIdx.x] = w[static_cast<size_t>(t) * k + threadIdx.x];
    }
    if (threadIdx.x == 0) rows[k] = k * T + t;
    __syncthreads();
    const int n4 = H / 4;
    for (int c = threadIdx.x; c < n4; c += blockDim.x) {
      float4 acc = accumulate ? reinterpret_cast<const float4*>(out + static_cast<size_t>(t) * H)[c]
                              : make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < k; ++j) {
        if (rows[j] < 0 || rows[j] >= (k + 1) * T) continue;  // a pair without a row
        const float4 v = reinterpret_cast<const float4*>(y + static_cast<size_t>(rows[j]) * H)[c];
        acc.x = fmaf(wt[j], v.x, acc.x);
        acc.y = fmaf(wt[j], v.y, acc.y);
        acc.z = fmaf(wt[j], v.z, acc.z);
        acc.w = fmaf(wt[j], v.w, acc.w);
      }
      const float4 v = reinterpret_cast<const float4*>(y + static_cast<size_t>(rows[k]) * H)[c];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
      reinterpret_cast<float4*>(out + static_cast<size_t>(t) * H)[c] = acc;
    }
  }
}

}  // namespace

cudaError_t launch_combine(const float* y_perm, const int32_t* row_of, const float* w, int T,
                           int H, int k, bool accumulate, float* out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = T < 152 * 8 ? T : 152 * 8;
  return launch_pdl(combine_kernel, dim3(blocks), dim3(256), 0, s, y_perm, row_of, w, T, H, k,
                    accumulate, out);
}

}  // namespace moe
