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
  pdl_launch_dependents();  // dependents wait for this grid's completion themselves
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
}

// ---------------------------------------------------------------- decode-size router
// Logits for up to a few hundred tokens are a GEMV-like product too small for
// the tensor-core pipeline to fill the GPU.  The reduction dimension is cut
// into slices so that every SM streams a slice of the router matrix at once:
// CTA (expert block, slice) stages its 32 router rows and the token rows of
// its slice as fp32 in shared memory (all global loads issued before the
// first use) and writes partial logits part[slice][t][e]; a second kernel
// adds the slices in slice order (a fixed order: the logits are the same on
// every run), adds the bias and selects the top-k, one warp per token.

constexpr int kPartExperts = 32;                 // router rows per CTA
constexpr int kPartTok = 64;                     // token rows per pass
constexpr int kPartRow = kRouterSliceK + 4;      // padded fp32 row: lanes on distinct banks
constexpr int kPartThreads = 256;                // warp w: experts 4w .. 4w + 3
constexpr int kPartWLoads = kPartExperts * (kRouterSliceK / 8) / kPartThreads;  // 4
constexpr int kPartXLoads = kPartTok * (kRouterSliceK / 8) / kPartThreads;      // 8
constexpr size_t kPartSmem = static_cast<size_t>(kPartTok + kPartExperts) * kPartRow * 4;

__device__ __forceinline__ void store_f32x8(float* dst, const uint4& v) {
  float f[8];
  bf16x8_to_f32(v, f);
  reinterpret_cast<float4*>(dst)[0] = make_float4(f[0], f[1], f[2], f[3]);
  reinterpret_cast<float4*>(dst)[1] = make_float4(f[4], f[5], f[6], f[7]);
}

// acc[a][e] = sum over the slice of x[lane + 32 a][k] * w[4 warp + e][k] for
// the first NR token rows of the lane (rows left out stay 0).
template <int NR>
__device__ __forceinline__ void partial_dot(const float* xs, const float* wsm, int lane, int warp,
                                            float (&acc)[2][4]) {
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[a][e] = 0.f;
  const float* xa = xs + lane * kPartRow;
  const float* xb = xs + (lane + 32) * kPartRow;
  const float* wb = wsm + (warp * 4) * kPartRow;
#pragma unroll 4
  for (int kk = 0; kk < kRouterSliceK; kk += 4) {
    float4 a4[2];
    a4[0] = *reinterpret_cast<const float4*>(xa + kk);
    if (NR == 2) a4[1] = *reinterpret_cast<const float4*>(xb + kk);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float4 b4 = *reinterpret_cast<const float4*>(wb + e * kPartRow + kk);
#pragma unroll
      for (int a = 0; a < NR; ++a) {
        acc[a][e] = fmaf(a4[a].x, b4.x, acc[a][e]);
        acc[a][e] = fmaf(a4[a].y, b4.y, acc[a][e]);
        acc[a][e] = fmaf(a4[a].z, b4.z, acc[a][e]);
        acc[a][e] = fmaf(a4[a].w, b4.w, acc[a][e]);
      }
    }
  }
}

// Clears n4 float4s of `out` with every thread of the grid (the layer's
// output when the down epilogue adds into it; null: nothing to clear).
__device__ __forceinline__ void clear_grid(float4* out, size_t n4) {
  if (!out) return;
  const size_t nthr = static_cast<size_t>(gridDim.x) * gridDim.y * blockDim.x;
  const size_t i0 = (static_cast<size_t>(blockIdx.y) * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
  for (size_t i = i0; i < n4; i += nthr) out[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// grid (ceil(E / 32), ceil(H / kRouterSliceK)), kPartThreads threads.
__global__ void __launch_bounds__(kPartThreads) router_partial_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr, int T, int H, int E,
    float* __restrict__ part, float4* __restrict__ zero_out, size_t zero_n4) {
  extern __shared__ float4 smem_f4[];
  float* xs = reinterpret_cast<float*>(smem_f4);  // [kPartTok][kPartRow]
  float* wsm = xs + kPartTok * kPartRow;          // [kPartExperts][kPartRow]
  const int e0 = blockIdx.x * kPartExperts;
  const int k0 = blockIdx.y * kRouterSliceK;
  const int nk = min(kRouterSliceK, H - k0);  // H % 8 == 0: whole 8-element chunks
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kChunksPerRow = kRouterSliceK / 8;
  pdl_wait();
  pdl_launch_dependents();  // dependents wait for this grid's completion themselves
  clear_grid(zero_out, zero_n4);
  // router rows of the block (zero past E and past H)
  uint4 wv[kPartWLoads];
#pragma unroll
  for (int j = 0; j < kPartWLoads; ++j) {
    const int i = threadIdx.x + j * kPartThreads, r = i / kChunksPerRow, c = i % kChunksPerRow;
    wv[j] = (e0 + r < E && c * 8 < nk)
                ? __ldg(reinterpret_cast<const uint4*>(wr + static_cast<size_t>(e0 + r) * H + k0) + c)
                : make_uint4(0u, 0u, 0u, 0u);
  }
  for (int t0 = 0; t0 < T; t0 += kPartTok) {
    const int nt = min(kPartTok, T - t0);
    uint4 xv[kPartXLoads];
#pragma unroll
    for (int j = 0; j < kPartXLoads; ++j) {
      const int i = threadIdx.x + j * kPartThreads, r = i / kChunksPerRow, c = i % kChunksPerRow;
      xv[j] = (r < nt && c * 8 < nk)
                  ? __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t0 + r) * H + k0) + c)
                  : make_uint4(0u, 0u, 0u, 0u);
    }
    if (t0 == 0) {
#pragma unroll
      for (int j = 0; j < kPartWLoads; ++j) {
        const int i = threadIdx.x + j * kPartThreads;
        store_f32x8(wsm + (i / kChunksPerRow) * kPartRow + (i % kChunksPerRow) * 8, wv[j]);
      }
    } else {
      __syncthreads();  // the previous pass has read xs
    }
#pragma unroll
    for (int j = 0; j < kPartXLoads; ++j) {
      const int i = threadIdx.x + j * kPartThreads;
      store_f32x8(xs + (i / kChunksPerRow) * kPartRow + (i % kChunksPerRow) * 8, xv[j]);
    }
    __syncthreads();
    // lane: tokens lane and lane + 32; warp: experts 4 warp .. 4 warp + 3
    float acc[2][4];
    if (nt > 32)
      partial_dot<2>(xs, wsm, lane, warp, acc);
    else
      partial_dot<1>(xs, wsm, lane, warp, acc);
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const int t = lane + 32 * a;
      if (t < nt) {
        float* dst = part + (static_cast<size_t>(blockIdx.y) * T + t0 + t) * E;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (e0 + warp * 4 + e < E) dst[e0 + warp * 4 + e] = acc[a][e];
      }
    }
  }
}

// One CTA per token, one thread per expert: z = (sum over slices, in slice
// order) + bias, with every slice's load in flight at once; warp 0 then
// selects the top-k from shared memory.  Writes idx / w, and z itself when
// z_out is given.
constexpr int kReduceBatch = 16;  // slice loads in flight per thread

__global__ void __launch_bounds__(kMaxE) router_reduce_topk_kernel(
    const float* __restrict__ part, const float* __restrict__ b, int T, int E, int slices, int k,
    int32_t* __restrict__ idx, float* __restrict__ w, float* __restrict__ z_out,
    const SmallPermOut perm) {
  __shared__ uint32_t keys_s[kMaxE];
  pdl_wait();
  pdl_launch_dependents();  // dependents wait for this grid's completion themselves
  const int t = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float acc = 0.f;
    for (int s0 = 0; s0 < slices; s0 += kReduceBatch) {
      float v[kReduceBatch];
#pragma unroll
      for (int j = 0; j < kReduceBatch; ++j)
        v[j] = s0 + j < slices ? part[(static_cast<size_t>(s0 + j) * T + t) * E + e] : 0.f;
#pragma unroll
      for (int j = 0; j < kReduceBatch; ++j)
        if (s0 + j < slices) acc += v[j];
    }
    const float zv = acc + b[e];
    keys_s[e] = float_key(zv);
    if (z_out) z_out[static_cast<size_t>(t) * E + e] = zv;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    uint32_t keys[kTopkVPL];
#pragma unroll
    for (int i = 0; i < kTopkVPL; ++i) {
      const int e = i * 32 + lane;
      keys[i] = e < E ? keys_s[e] : 0u;
    }
    int e;
    float wv;
    warp_topk_keys(keys, E, k, &e, &wv);
    if (lane < k) {
      idx[static_cast<size_t>(t) * k + lane] = e;
      w[static_cast<size_t>(t) * k + lane] = wv;
    }
  }
  if (perm.done) {
    // the last CTA to finish runs the permutation over every token's selection
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(perm.done, 1) == static_cast<int>(gridDim.x) - 1;
    __syncthreads();
    if (s_last) {
      __threadfence();
      small_permutation(idx, w, T, E, k, perm.BN, perm.offsets, perm.gather, perm.row_of,
                        perm.roww, perm.table, perm.table2, perm.BN2);
      if (threadIdx.x == 0) *perm.done = 0;
    }
  }
}

// One warp per token: top-k, sigmoid, renormalisation.
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ z, int T, int E,
                                                   int k, int32_t* __restrict__ idx,
                                                   float* __restrict__ w,
                                                   float4* __restrict__ zero_out,
                                                   size_t zero_n4) {
  pdl_wait();
  pdl_launch_dependents();  // dependents wait for this grid's completion themselves
  clear_grid(zero_out, zero_n4);
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
}


// ---------------------------------------------------------------- one-launch routing, T <= 16
// At decode sizes the routing is a chain of latencies, not of bytes (2.36 MB
// of router weights): one launch does all of it.  CTA = 2 experts x 4 warps;
// warp (e, q) covers quarter q of the reduction for expert e, every lane
// issuing its router loads (and a batch of four tokens' x loads) before the
// first use; the quarters are added in a fixed order with the bias, so the
// logits are the same bits on every run.  The last CTA to finish (a counter
// in the workspace, zero between calls) selects the top-k of every token,
// one warp per token, and builds the permutation in shared memory: with at
// most 16 x 16 (token, slot) pairs, counts and ranks are read off the pairs
// directly, and one block-wide scan gives the tile table.

constexpr int kRsExperts = 2;                           // experts per CTA
constexpr int kRsSplit = 4;                             // warps per expert (reduction quarters)
constexpr int kRsThreads = 32 * kRsExperts * kRsSplit;  // 256
constexpr int kRsChunks = 4;                            // 16-byte chunks per lane (H <= 4096)
constexpr int kRsTokBatch = 4;                          // tokens whose x loads are in flight together

// Exclusive scan of v[0..n) in shared memory by the whole CTA (n <= 1024:
// each warp scans 32-element chunks, warp 0 scans the chunk sums); *total
// gets the sum.  Every thread calls it; it synchronises before it returns.
__device__ __forceinline__ void block_exclusive_scan(int* v, int n, int* total) {
  __shared__ int chunk_sum[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int nchunks = (n + 31) >> 5;
  for (int c = warp; c < nchunks; c += nw) {
    const int i = c * 32 + lane;
    const int x = i < n ? v[i] : 0;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (i < n) v[i] = incl - x;
    if (lane == 31) chunk_sum[c] = incl;
  }
  __syncthreads();
  if (warp == 0) {
    const int x = lane < nchunks ? chunk_sum[lane] : 0;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane < nchunks) chunk_sum[lane] = incl - x;
    if (lane == 31) *total = incl;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) v[i] += chunk_sum[i >> 5];
  __syncthreads();
}

// Tile table of groups 0..E (counts from the offsets off[0..E+1]): entries
// of at most BN rows, in group order.
__device__ __forceinline__ void small_tile_table(const int* off, int* ntile, int E, int BN,
                                                 int32_t* __restrict__ table) {
  __shared__ int n_entries;
  for (int g = threadIdx.x; g <= E; g += blockDim.x) ntile[g] = (off[g + 1] - off[g] + BN - 1) / BN;
  __syncthreads();
  block_exclusive_scan(ntile, E + 1, &n_entries);
  TileEntry* ent = reinterpret_cast<TileEntry*>(reinterpret_cast<char*>(table) + kTableHeaderBytes);
  for (int g = threadIdx.x; g <= E; g += blockDim.x) {
    const int o = off[g], c = off[g + 1] - o;
    for (int i = 0, r = 0; r < c; ++i, r += BN) {
      TileEntry te;
      te.group = g;
      te.row0 = o + r;
      te.nrows = min(BN, c - r);
      te.ntiles = (c + BN - 1) / BN;
      ent[ntile[g] + i] = te;
    }
  }
  if (threadIdx.x == 0) table[0] = n_entries;
  __syncthreads();
}

__global__ void __launch_bounds__(kRsThreads) route_small_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr, const float* __restrict__ b,
    int T, int H, int E, int k, float* __restrict__ z, int32_t* __restrict__ idx,
    float* __restrict__ w, const SmallPermOut perm, float4* __restrict__ zero_out,
    size_t zero_n4) {
  __shared__ float red[kRsExperts][kRsSplit][kRouteSmallT];
  __shared__ int s_last;
  pdl_wait();
  pdl_launch_dependents();  // dependents wait for this grid's completion themselves
  clear_grid(zero_out, zero_n4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int el = warp / kRsSplit, q = warp % kRsSplit;
  const int e = blockIdx.x * kRsExperts + el;
  const int cq = H / (8 * kRsSplit);  // 16-byte chunks per quarter (H % 128 == 0)
  if (e < E) {
    const uint4* wrow = reinterpret_cast<const uint4*>(wr + static_cast<size_t>(e) * H) + q * cq;
    uint4 wv[kRsChunks];
#pragma unroll
    for (int i = 0; i < kRsChunks; ++i) {
      const int c = lane + 32 * i;
      wv[i] = c < cq ? __ldg(wrow + c) : make_uint4(0u, 0u, 0u, 0u);
    }
    for (int t0 = 0; t0 < T; t0 += kRsTokBatch) {
      uint4 xv[kRsTokBatch][kRsChunks];
#pragma unroll
      for (int tt = 0; tt < kRsTokBatch; ++tt) {
        const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t0 + tt) * H) + q * cq;
#pragma unroll
        for (int i = 0; i < kRsChunks; ++i) {
          const int c = lane + 32 * i;
          xv[tt][i] = (t0 + tt < T && c < cq) ? __ldg(xr + c) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int tt = 0; tt < kRsTokBatch; ++tt) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < kRsChunks; ++i) {
          float xf[8], wf[8];
          bf16x8_to_f32(xv[tt][i], xf);
          bf16x8_to_f32(wv[i], wf);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc = fmaf(xf[j], wf[j], acc);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0 && t0 + tt < T) red[el][q][t0 + tt] = acc;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < kRsExperts * kRouteSmallT) {
    const int e2 = blockIdx.x * kRsExperts + threadIdx.x / kRouteSmallT;
    const int t = threadIdx.x % kRouteSmallT;
    const int l2 = threadIdx.x / kRouteSmallT;
    if (e2 < E && t < T)
      z[static_cast<size_t>(t) * E + e2] =
          ((red[l2][0][t] + red[l2][1][t]) + (red[l2][2][t] + red[l2][3][t])) + b[e2];
  }
  // The last CTA to finish selects and permutes.  The CTA's logits are
  // ordered before its count by the barrier and the counting thread's
  // release; the last CTA's acquire orders its reads of every CTA's logits
  // after their counts.
  __syncthreads();
  if (threadIdx.x == 0)
    s_last = atom_acq_rel_gpu_add(perm.done, 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (!s_last) return;

  __shared__ int s_e[kRouteSmallT * kMaxTopK];
  __shared__ float s_w[kRouteSmallT * kMaxTopK];
  __shared__ int s_off[kMaxE + 2];
  __shared__ int s_nt[kMaxE + 1];
  __shared__ int s_total;
  const int P = T * k;
  for (int t = warp; t < T; t += kRsThreads / 32) {
    uint32_t keys[kTopkVPL];
    const float* zr = z + static_cast<size_t>(t) * E;
#pragma unroll
    for (int i = 0; i < kTopkVPL; ++i) {
      const int ee = i * 32 + lane;
      keys[i] = ee < E ? float_key(__ldcg(zr + ee)) : 0u;
    }
    int ew;
    float wv;
    warp_topk_keys(keys, E, k, &ew, &wv);
    if (lane < k) {
      s_e[t * k + lane] = ew;
      s_w[t * k + lane] = wv;
      idx[static_cast<size_t>(t) * k + lane] = ew;
      w[static_cast<size_t>(t) * k + lane] = wv;
    }
  }
  __syncthreads();
  if (T <= perm.BN && (!perm.table2 || T <= perm.BN2)) {
    // Every routed group holds at most T <= BN rows, one tile entry each.  A
    // pair's row is its rank in (expert, token) order: the pairs of smaller
    // experts, then this expert's pairs of earlier tokens (a token's ids are
    // distinct, so pair order is token order within an expert), counted over
    // the at most kRouteSmallT * k pairs; offsets are binary searches in the
    // sorted experts and the entries their runs.  No scan, two barriers.
    __shared__ int s_sorted[kRouteSmallT * kMaxTopK];  // expert of row r < P
    for (int p = threadIdx.x; p < P; p += kRsThreads) {
      const int ee = s_e[p];
      int r = 0;
      for (int q = 0; q < P; ++q) {
        const int eq = s_e[q];
        r += (eq < ee) || (eq == ee && q < p);
      }
      s_sorted[r] = ee;
      perm.gather[r] = p / k;
      perm.row_of[p] = r;
      perm.roww[r] = s_w[p];
    }
    for (int t = threadIdx.x; t < T; t += kRsThreads) {
      perm.gather[P + t] = t;
      perm.roww[P + t] = 1.0f;
    }
    __syncthreads();
    for (int g = threadIdx.x; g <= E + 1; g += kRsThreads) {
      int lo = 0, hi = P;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s_sorted[mid] < g) lo = mid + 1;
        else hi = mid;
      }
      perm.offsets[g] = g <= E ? lo : P + T;  // the shared group E: rows P .. P + T
    }
    TileEntry* ent = reinterpret_cast<TileEntry*>(reinterpret_cast<char*>(perm.table) +
                                                  kTableHeaderBytes);
    TileEntry* ent2 = perm.table2 ? reinterpret_cast<TileEntry*>(
                                        reinterpret_cast<char*>(perm.table2) + kTableHeaderBytes)
                                  : nullptr;
    for (int r = threadIdx.x; r < P; r += kRsThreads) {
      const int ee = s_sorted[r];
      if (r > 0 && s_sorted[r - 1] == ee) continue;  // not the first row of its group
      int run = 0, end = r + 1;
      for (int q = 1; q <= r; ++q) run += s_sorted[q] != s_sorted[q - 1];
      while (end < P && s_sorted[end] == ee) ++end;
      const TileEntry te{ee, r, end - r, 1};
      ent[run] = te;
      if (ent2) ent2[run] = te;
    }
    if (threadIdx.x == 0) {
      int runs = P > 0 ? 1 : 0;
      for (int q = 1; q < P; ++q) runs += s_sorted[q] != s_sorted[q - 1];
      const TileEntry te{E, P, T, 1};
      ent[runs] = te;
      perm.table[0] = runs + 1;
      if (ent2) {
        ent2[runs] = te;
        perm.table2[0] = runs + 1;
      }
      *perm.done = 0;
    }
    return;
  }
  for (int g = threadIdx.x; g <= E; g += kRsThreads) s_off[g] = 0;
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += kRsThreads) atomicAdd(&s_off[s_e[p]], 1);
  if (threadIdx.x == 0) s_off[E] = T;  // the shared expert: every token
  __syncthreads();
  block_exclusive_scan(s_off, E + 1, &s_total);
  if (threadIdx.x == 0) s_off[E + 1] = s_total;
  __syncthreads();
  for (int g = threadIdx.x; g <= E + 1; g += kRsThreads) perm.offsets[g] = s_off[g];
  // rank of a pair among the earlier pairs of its expert (a token's ids are
  // distinct, so earlier pairs of an expert belong to earlier tokens)
  for (int p = threadIdx.x; p < P; p += kRsThreads) {
    const int ee = s_e[p];
    int rank = 0;
    for (int p2 = 0; p2 < p; ++p2) rank += s_e[p2] == ee;
    const int r = s_off[ee] + rank, t = p / k;
    perm.gather[r] = t;
    perm.row_of[p] = r;
    perm.roww[r] = s_w[p];
  }
  for (int t = threadIdx.x; t < T; t += kRsThreads) {
    perm.gather[P + t] = t;
    perm.roww[P + t] = 1.0f;
  }
  small_tile_table(s_off, s_nt, E, perm.BN, perm.table);
  if (perm.table2) small_tile_table(s_off, s_nt, E, perm.BN2, perm.table2);
  if (threadIdx.x == 0) *perm.done = 0;
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

cudaError_t launch_router_partials(const uint16_t* x, const uint16_t* w_router, float* part,
                                  int T, int H, int E, float* zero_out, size_t zero_n,
                                  cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  cudaError_t err = cudaFuncSetAttribute(router_partial_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kPartSmem));
  if (err != cudaSuccess) return err;
  const dim3 grid((E + kPartExperts - 1) / kPartExperts, router_slices(H));
  return launch_pdl(router_partial_kernel, grid, dim3(kPartThreads), kPartSmem, s, x, w_router,
                    T, H, E, part, reinterpret_cast<float4*>(zero_out), zero_n / 4);
}

cudaError_t launch_route_small(const uint16_t* x, const uint16_t* w_router, const float* b, int T,
                               int H, int E, int k, float* z, int32_t* idx, float* w,
                               const SmallPermOut& perm, float* zero_out, size_t zero_n,
                               cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (T > kRouteSmallT || H > kRsChunks * 32 * 8 * kRsSplit || !perm.done)
    return cudaErrorInvalidValue;
  return launch_pdl(route_small_kernel, dim3((E + kRsExperts - 1) / kRsExperts), dim3(kRsThreads),
                    0, s, x, w_router, b, T, H, E, k, z, idx, w, perm,
                    reinterpret_cast<float4*>(zero_out), zero_n / 4);
}

cudaError_t launch_router_reduce_topk(const float* part, const float* b, int T, int H, int E,
                                      int k, int32_t* idx, float* w, float* z,
                                      const SmallPermOut* perm, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (perm && T > kSmallT) return cudaErrorInvalidValue;
  const SmallPermOut none{};
  const int threads = ((E + 31) / 32) * 32;  // E <= kMaxE
  return launch_pdl(router_reduce_topk_kernel, dim3(T), dim3(threads), 0, s, part, b, T, E,
                    router_slices(H), k, idx, w, z, perm ? *perm : none);
}

cudaError_t launch_topk(const float* z, int T, int E, int k, int32_t* idx, float* w,
                        cudaStream_t s, float* zero_out, size_t zero_n) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(topk_kernel, dim3((T + 7) / 8), dim3(256), 0, s, z, T, E, k, idx, w,
                    reinterpret_cast<float4*>(zero_out), zero_n / 4);
}

}  // namespace moe
