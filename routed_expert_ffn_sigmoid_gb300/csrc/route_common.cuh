// Device building blocks shared by the router and permutation kernels: the
// warp top-k of one token's logits and a warp-0 exclusive scan.
#pragma once

#include <stdint.h>

#include "moe_kernels.h"

namespace moe {

// Order-preserving map of a float onto uint32 (larger float -> larger key).
// -0 and +0 compare equal as floats, so both map to the key of +0: a tie
// between them is then decided by the expert index like any other tie.
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

constexpr int kTopkVPL = kMaxE / 32;  // logits held per lane

// Top-k of one token's E logits by one warp ("Top-8 expert selection",
// sigmoid routing and "Weight normalization": "Add GLM-5.3-Flash (glm5next)
// support with ROCmFP mix qtypes (105/106)", section "MoE FFN (REAL routed
// expert execution)"; ties to the lower index: deterministic top-k, "feat(glm53):
// add device-resident HIP backend for MI350P", "Key changes").
// Lane L holds experts L, L+32, ...  Each round, every lane takes its largest
// remaining key (the first of equal keys: its lowest expert), the warp takes
// the largest of those with one 32-bit max reduction, and the lowest expert
// holding it with one min reduction: the larger score wins and an exact tie
// goes to the lower expert index.  Lane j < k ends with slot j: *e_out, and
// *w_out = sigmoid(z_j) / sum of the k sigmoids.  keys[i] = float_key(z) of
// expert i * 32 + lane (any value where that expert does not exist).
__device__ __forceinline__ void warp_topk_keys(const uint32_t (&keys)[kTopkVPL], int E, int k,
                                               int* e_out, float* w_out) {
  const int lane = threadIdx.x & 31;
  const int nv = (E + 31) >> 5;  // key slots in use (warp-uniform)
  uint32_t taken = 0;
  int my_e = 0;
  float my_z = 0.f;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0;  // below every key of a float (float_key of -inf is 0x007FFFFF)
    uint32_t be = 0xFFFFFFFFu;
#pragma unroll
    for (int i = 0; i < kTopkVPL; ++i) {
      if (i >= nv) break;
      const int e = i * 32 + lane;
      if (e < E && !((taken >> i) & 1u) && keys[i] > bk) {
        bk = keys[i];
        be = static_cast<uint32_t>(e);
      }
    }
    const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
    const int e_win = static_cast<int>(__reduce_min_sync(0xffffffffu, bk == mk ? be : 0xFFFFFFFFu));
    if ((e_win & 31) == lane) taken |= 1u << (e_win >> 5);
    if (lane == j) {
      my_e = e_win;
      my_z = key_float(mk);
    }
  }
  const float s = lane < k ? 1.0f / (1.0f + expf(-my_z)) : 0.f;
  float sum = s;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  *e_out = my_e;
  *w_out = s / sum;
}

// The same selection from a row of E logits in memory.
__device__ __forceinline__ void warp_topk(const float* __restrict__ zr, int E, int k, int* e_out,
                                          float* w_out) {
  const int lane = threadIdx.x & 31;
  uint32_t keys[kTopkVPL];
#pragma unroll
  for (int i = 0; i < kTopkVPL; ++i) {
    const int e = i * 32 + lane;
    keys[i] = e < E ? float_key(zr[e]) : 0u;
  }
  warp_topk_keys(keys, E, k, e_out, w_out);
}

// Exclusive scan of n values in shared memory by warp 0; *total gets the sum.
// Other threads return at once; the caller synchronises.
__device__ __forceinline__ void warp0_exclusive_scan(int* v, int n, int* total) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  int carry = 0;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    const int x = i < n ? v[i] : 0;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (i < n) v[i] = carry + incl - x;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) *total = carry;
}

__device__ __forceinline__ void write_tile_table(const int* off, int* ntile, int E, int BN,
                                                 int* n_entries, int32_t* __restrict__ table) {
  for (int g = threadIdx.x; g <= E; g += blockDim.x) ntile[g] = (off[g + 1] - off[g] + BN - 1) / BN;
  __syncthreads();
  warp0_exclusive_scan(ntile, E + 1, n_entries);
  __syncthreads();
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
  if (threadIdx.x == 0) table[0] = *n_entries;
}

// Decode-size permutation by one CTA (T <= kSmallT tokens, any block size
// that is a multiple of 32): from the top-k selection idx / w [T][k] in
// global memory, the expert histogram, exclusive offsets (the shared expert
// appended as group E), stable ranks from per-expert token bitmaps,
// gather / row_of / row weights and the tile table -- the work of the count,
// scan and scatter kernels with no launch in between, with the same results.
// The selection may have been written by other CTAs of the calling grid: it
// is read past L1.  As in the multi-kernel path, an id outside [0, E) gets no
// row (row_of = -1) and is left out of the counts; with w == nullptr no row
// weights are written (roww may then be null too).
__device__ __forceinline__ void small_permutation(const int32_t* idx, const float* w, int T, int E,
                                                  int k, int BN, int32_t* __restrict__ offsets,
                                                  int32_t* __restrict__ gather,
                                                  int32_t* __restrict__ row_of,
                                                  float* __restrict__ roww,
                                                  int32_t* __restrict__ table,
                                                  int32_t* __restrict__ table2 = nullptr,
                                                  int BN2 = 0) {
  __shared__ int s_idx[kSmallT * kMaxTopK];
  __shared__ float s_w[kSmallT * kMaxTopK];
  __shared__ int cnt[kMaxE + 2];
  __shared__ int ntile[kMaxE + 1];
  __shared__ uint32_t bits[kMaxE][kSmallT / 32];
  __shared__ int total_rows, n_entries;
  for (int g = threadIdx.x; g <= E; g += blockDim.x) cnt[g] = 0;
  for (int i = threadIdx.x; i < E * (kSmallT / 32); i += blockDim.x) (&bits[0][0])[i] = 0u;
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    s_idx[i] = __ldcg(idx + i);
    s_w[i] = w ? __ldcg(w + i) : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    const int t = i / k, e = s_idx[i];
    if (e < 0 || e >= E) continue;  // out-of-range ids are ignored
    atomicAdd(&cnt[e], 1);
    atomicOr(&bits[e][t >> 5], 1u << (t & 31));
  }
  __syncthreads();
  if (threadIdx.x == 0) cnt[E] = T;
  __syncthreads();
  warp0_exclusive_scan(cnt, E + 1, &total_rows);  // cnt becomes the offsets
  __syncthreads();
  if (threadIdx.x == 0) cnt[E + 1] = total_rows;
  __syncthreads();
  for (int g = threadIdx.x; g <= E + 1; g += blockDim.x) offsets[g] = cnt[g];
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    const int t = i / k, e = s_idx[i];
    if (e < 0 || e >= E) {  // an out-of-range id gets no row
      row_of[i] = -1;
      continue;
    }
    int rank = __popc(bits[e][t >> 5] & ((1u << (t & 31)) - 1u));
    for (int wd = 0; wd < (t >> 5); ++wd) rank += __popc(bits[e][wd]);
    const int r = cnt[e] + rank;
    gather[r] = t;
    row_of[i] = r;
    if (w) roww[r] = s_w[i];
  }
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    gather[k * T + t] = t;
    if (w) roww[k * T + t] = 1.0f;
  }
  write_tile_table(cnt, ntile, E, BN, &n_entries, table);
  if (table2) {
    __syncthreads();  // ntile is reused
    write_tile_table(cnt, ntile, E, BN2, &n_entries, table2);
  }
}

// Launch helper: programmatic stream serialization lets a kernel begin while
// its predecessor drains; every kernel launched this way calls pdl_wait()
// before it touches data a predecessor produced.  The routing kernels call
// pdl_launch_dependents() right after that wait: the next grid's CTAs are
// then scheduled while this one runs (hiding their launch), and still wait
// in their own pdl_wait() for this grid to complete.
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace moe
