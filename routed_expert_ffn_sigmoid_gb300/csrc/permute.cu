// Counting-sort permutation of (token, slot) pairs by expert.
//
// The grouping the per-expert matmuls run on ("ggml_mul_mat_id" for gate, up
// and down in "Add GLM-5.3-Flash (glm5next) support with ROCmFP mix qtypes
// (105/106)", section "MoE FFN (REAL routed expert execution)"), built as a
// stable counting sort so that rows of one expert are ordered by token:
//   1. per 128-token block, a shared-memory histogram of expert ids;
//   2. one CTA turns the block histograms into per-block row bases and the
//      exclusive offsets (the shared expert appended as group E with all T
//      tokens), and cuts every group into tiles of at most BN rows;
//   3. per block, a token bitmap per expert gives each pair its rank among
//      the block's earlier tokens -> row = base + rank;
//   4. x rows are gathered into permuted order with 16-byte loads.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "moe_kernels.h"
#include "ptx.cuh"
#include "route_common.cuh"

namespace moe {
namespace {

constexpr int kWordsPerBlock = kPermTokBlock / 32;

__global__ void __launch_bounds__(256) perm_count_kernel(const int32_t* __restrict__ idx, int T,
                                                         int E, int k,
                                                         int32_t* __restrict__ blockcnt) {
  __shared__ int cnt[kMaxE];
  pdl_wait();
  pdl_launch_dependents();  // dependents wait for this grid's completion themselves
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int t0 = blockIdx.x * kPermTokBlock;
  const int nt = min(kPermTokBlock, T - t0);
  const int32_t* ib = idx + static_cast<size_t>(t0) * k;
  for (int i = threadIdx.x; i < nt * k; i += blockDim.x) {
    const int e = ib[i];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);  // out-of-range ids are ignored
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    blockcnt[static_cast<size_t>(blockIdx.x) * E + e] = cnt[e];
}

// One CTA of 1024 threads.
__global__ void __launch_bounds__(1024) perm_scan_kernel(int32_t* __restrict__ blockcnt, int T,
                                                         int E, int k,
                                                         int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ table, int BN) {
  __shared__ int tot[kMaxE + 1];
  __shared__ int off[kMaxE + 2];
  __shared__ int ntile[kMaxE + 1];
  __shared__ int n_entries;
  __shared__ int total_rows;
  pdl_wait();
  pdl_launch_dependents();  // dependents wait for this grid's completion themselves
  const int nblk = (T + kPermTokBlock - 1) / kPermTokBlock;
  // per expert: running sum over blocks (becomes the block-relative base)
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int b = 0; b < nblk; ++b) {
      const size_t p = static_cast<size_t>(b) * E + e;
      const int c = blockcnt[p];
      blockcnt[p] = run;
      run += c;
    }
    tot[e] = run;
  }
  if (threadIdx.x == 0) tot[E] = T;
  __syncthreads();
  for (int g = threadIdx.x; g <= E; g += blockDim.x) off[g] = tot[g];
  __syncthreads();
  warp0_exclusive_scan(off, E + 1, &total_rows);
  __syncthreads();
  if (threadIdx.x == 0) off[E + 1] = total_rows;
  __syncthreads();
  for (int g = threadIdx.x; g <= E + 1; g += blockDim.x) offsets[g] = off[g];
  // block bases become absolute rows
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    for (int b = 0; b < nblk; ++b) blockcnt[static_cast<size_t>(b) * E + e] += off[e];
  // tile table: group g is cut into ceil(cnt / BN) entries
  for (int g = threadIdx.x; g <= E; g += blockDim.x) ntile[g] = (tot[g] + BN - 1) / BN;
  __syncthreads();
  warp0_exclusive_scan(ntile, E + 1, &n_entries);
  __syncthreads();
  TileEntry* ent = reinterpret_cast<TileEntry*>(reinterpret_cast<char*>(table) + kTableHeaderBytes);
  for (int g = threadIdx.x; g <= E; g += blockDim.x) {
    const int c = tot[g];
    for (int i = 0, r = 0; r < c; ++i, r += BN) {
      TileEntry te;
      te.group = g;
      te.row0 = off[g] + r;
      te.nrows = min(BN, c - r);
      te.ntiles = (c + BN - 1) / BN;
      ent[ntile[g] + i] = te;
    }
  }
  if (threadIdx.x == 0) table[0] = n_entries;
}

__global__ void __launch_bounds__(256) perm_scatter_kernel(const int32_t* __restrict__ idx,
                                                           const float* __restrict__ w,
                                                           const int32_t* __restrict__ blockbase,
                                                           int T, int E, int k,
                                                           int32_t* __restrict__ gather,
                                                           int32_t* __restrict__ row_of,
                                                           float* __restrict__ roww) {
  __shared__ uint32_t bits[kMaxE][kWordsPerBlock];
  pdl_wait();
  pdl_launch_dependents();  // dependents wait for this grid's completion themselves
  for (int i = threadIdx.x; i < E * kWordsPerBlock; i += blockDim.x) (&bits[0][0])[i] = 0u;
  __syncthreads();
  const int t0 = blockIdx.x * kPermTokBlock;
  const int nt = min(kPermTokBlock, T - t0);
  const int32_t* ib = idx + static_cast<size_t>(t0) * k;
  for (int i = threadIdx.x; i < nt * k; i += blockDim.x) {
    const int tl = i / k;
    const int e = ib[i];
    if (e >= 0 && e < E) atomicOr(&bits[e][tl >> 5], 1u << (tl & 31));
  }
  __syncthreads();
  const int32_t* base = blockbase + static_cast<size_t>(blockIdx.x) * E;
  for (int i = threadIdx.x; i < nt * k; i += blockDim.x) {
    const int tl = i / k;
    const int e = ib[i];
    if (e < 0 || e >= E) {  // an out-of-range id gets no row
      row_of[static_cast<size_t>(t0) * k + i] = -1;
      continue;
    }
    int rank = __popc(bits[e][tl >> 5] & ((1u << (tl & 31)) - 1u));
    for (int wd = 0; wd < (tl >> 5); ++wd) rank += __popc(bits[e][wd]);
    const int r = base[e] + rank;
    const int t = t0 + tl;
    gather[r] = t;
    row_of[static_cast<size_t>(t0) * k + i] = r;
    if (roww) roww[r] = w[static_cast<size_t>(t0) * k + i];
  }
  // the shared expert's rows: every token, in order, after the routed rows
  for (int tl = threadIdx.x; tl < nt; tl += blockDim.x) {
    const int r = k * T + t0 + tl;
    gather[r] = t0 + tl;
    if (roww) roww[r] = 1.0f;
  }
}

// Token rows into x_perm, one warp per (token, column segment), grid-stride:
// each piece of x[t] is read once and written to the token's k routed rows
// (row_of[t][j]) and to its shared row k*T + t -- in token order, so each
// source row crosses HBM once even when x is larger than L2 (a copy in row
// order re-reads it up to k+1 times); `segs` segments per row keep enough
// warps busy when T is small.  H is a multiple of 128, so a row is a whole
// number of 16-byte chunks.  When zero_out is set, the kernel also clears
// the layer output (zero_n4 float4s) that the down kernel later adds into.
template <bool kToFp16>
__global__ void __launch_bounds__(256) scatter_rows_kernel(const uint16_t* __restrict__ x,
                                                           const int32_t* __restrict__ row_of,
                                                           int T, int H, int k, int segs,
                                                           uint16_t* __restrict__ x_perm,
                                                           float4* __restrict__ zero_out,
                                                           size_t zero_n4) {
  pdl_wait();
  pdl_launch_dependents();  // dependents wait for this grid's completion themselves
  if (zero_out) {
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < zero_n4;
         i += stride)
      zero_out[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int seg_chunks = H / 8 / segs;
  const int rows = (k + 1) * T;
  for (int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; item < T * segs; item += warps) {
    const int t = item / segs, c0 = (item % segs) * seg_chunks;
    uint4* dst[kMaxTopK + 1];
#pragma unroll
    for (int j = 0; j <= kMaxTopK; ++j) {
      // a row outside the buffer (row_of = -1: an out-of-range expert id) is
      // clamped into it, so the write stays in bounds; the rows' contents are
      // then as undefined as the results are for such ids
      const int r = j < k ? min(max(row_of[static_cast<size_t>(t) * k + j], 0), rows - 1)
                          : k * T + t;
      dst[j] = reinterpret_cast<uint4*>(x_perm + static_cast<size_t>(r) * H);
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
    for (int c = c0 + lane; c < c0 + seg_chunks; c += 32) {
      uint4 v = __ldg(src + c);
      if (kToFp16) {
        // bf16 -> fp16 (exact in fp16's normal range), the 8 columns stored
        // in the Int4 kernels' operand order 0, 4, 1, 5, 2, 6, 3, 7
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
        float e[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          e[2 * i] = __uint_as_float(wv[i] << 16);
          e[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
        }
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half2 h2 = __floats2half2_rn(e[i], e[i + 4]);
          o[i] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        v = make_uint4(o[0], o[1], o[2], o[3]);
      }
#pragma unroll
      for (int j = 0; j <= kMaxTopK; ++j)
        if (j <= k) dst[j][c] = v;
    }
  }
}

// One CTA per token: the row maximum |x| gives sigma = 2^(8 - e) with
// max = f 2^e, f in [0.5, 1), so max |x sigma| lies in [128, 256), inside
// e4m3's range (448).  hi = e4m3(x sigma) and lo = e4m3(x sigma - hi),
// both rounded to nearest by the hardware conversion; x sigma is exact (a
// bf16 value times a power of two) and so is x sigma - hi in fp32.  The two
// planes go to each of the token's k + 1 permuted rows, each aligned group
// of 8 elements in the order (0, 1, 4, 5, 2, 3, 6, 7).
constexpr int kSplitThreads = 256;

__global__ void __launch_bounds__(kSplitThreads) split_rows_e4m3_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ row_of, int T, int H, int k,
    uint8_t* __restrict__ x8, float* __restrict__ xinv, float4* __restrict__ zero_out,
    size_t zero_n4) {
  __shared__ float s_max[kSplitThreads / 32];
  __shared__ int32_t s_rows[kMaxTopK + 1];
  pdl_wait();
  pdl_launch_dependents();  // dependents wait for this grid's completion themselves
  if (zero_out) {
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < zero_n4;
         i += stride)
      zero_out[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int chunks = H / 8;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
    if (threadIdx.x <= k)
      s_rows[threadIdx.x] =
          threadIdx.x < k ? row_of[static_cast<size_t>(t) * k + threadIdx.x] : k * T + t;
    float mx = 0.f;
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
      const uint4 v = __ldg(src + c);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(wv[i] << 16)),
                             fabsf(__uint_as_float(wv[i] & 0xFFFF0000u))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_max[warp] = mx;
    __syncthreads();
    mx = 0.f;
#pragma unroll
    for (int i = 0; i < kSplitThreads / 32; ++i) mx = fmaxf(mx, s_max[i]);
    int e = 0;
    if (mx > 0.f) frexpf(mx, &e);
    e = max(e, -100);  // a row of zeros (or tiny values) keeps a finite scale
    const float sigma = ldexpf(1.0f, 8 - e);
    if (threadIdx.x <= k) xinv[s_rows[threadIdx.x]] = 1.0f / sigma;
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
      const uint4 v = __ldg(src + c);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      uint32_t hi[2] = {0u, 0u}, lo[2] = {0u, 0u};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float y =
            __uint_as_float((i & 1) ? (wv[i >> 1] & 0xFFFF0000u) : (wv[i >> 1] << 16)) * sigma;
        const __nv_fp8_storage_t h8 = __nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3);
        const float hf = __half2float(__half(__nv_cvt_fp8_to_halfraw(h8, __NV_E4M3)));
        const __nv_fp8_storage_t l8 = __nv_cvt_float_to_fp8(y - hf, __NV_SATFINITE, __NV_E4M3);
        // element i goes to byte position (0, 1, 4, 5, 2, 3, 6, 7)[i], the
        // order in which the 8-bit GEMM's dequantisers emit the weights
        const int pos = (i & 1) | ((i & 2) << 1) | ((i & 4) >> 1);
        hi[pos >> 2] |= static_cast<uint32_t>(h8) << (8 * (pos & 3));
        lo[pos >> 2] |= static_cast<uint32_t>(l8) << (8 * (pos & 3));
      }
      for (int j = 0; j <= k; ++j) {
        uint8_t* rowp = x8 + static_cast<size_t>(s_rows[j]) * 2 * H;
        reinterpret_cast<uint2*>(rowp)[c] = make_uint2(hi[0], hi[1]);
        reinterpret_cast<uint2*>(rowp + H)[c] = make_uint2(lo[0], lo[1]);
      }
    }
    __syncthreads();  // s_rows and s_max are rewritten for the next token
  }
}

// Tile table from an offsets array (E+2 entries), one CTA.  Offsets are
// clamped into [0, rows] and made non-decreasing, and no more than
// `capacity` entries are written, so inconsistent offsets cannot send a tile
// outside the row range or the table outside its buffer.
__global__ void __launch_bounds__(1024) table_from_offsets_kernel(const int32_t* __restrict__ offsets,
                                                                  int E, int rows, int capacity,
                                                                  int32_t* __restrict__ table,
                                                                  int BN) {
  __shared__ int lo[kMaxE + 1];
  __shared__ int ntile[kMaxE + 1];
  __shared__ int n_entries;
  pdl_wait();
  pdl_launch_dependents();  // dependents wait for this grid's completion themselves
  for (int g = threadIdx.x; g <= E; g += blockDim.x) {
    const int a = min(max(offsets[g], 0), rows);
    const int b = min(max(offsets[g + 1], a), rows);
    lo[g] = a;
    ntile[g] = (b - a + BN - 1) / BN;
  }
  __syncthreads();
  warp0_exclusive_scan(ntile, E + 1, &n_entries);
  __syncthreads();
  TileEntry* ent = reinterpret_cast<TileEntry*>(reinterpret_cast<char*>(table) + kTableHeaderBytes);
  for (int g = threadIdx.x; g <= E; g += blockDim.x) {
    const int o = lo[g];
    const int c = min(max(offsets[g + 1], o), rows) - o;
    for (int i = 0, r = 0; r < c; ++i, r += BN) {
      if (ntile[g] + i >= capacity) break;
      TileEntry te;
      te.group = g;
      te.row0 = o + r;
      te.nrows = min(BN, c - r);
      te.ntiles = (c + BN - 1) / BN;
      ent[ntile[g] + i] = te;
    }
  }
  if (threadIdx.x == 0) table[0] = min(n_entries, capacity);
}

}  // namespace

namespace {

// The decode-size permutation as a launch of its own (one CTA).
__global__ void __launch_bounds__(kSmallThreads) small_permutation_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ w, int T, int E, int k, int BN,
    int32_t* __restrict__ offsets, int32_t* __restrict__ gather, int32_t* __restrict__ row_of,
    float* __restrict__ roww, int32_t* __restrict__ table, int32_t* __restrict__ table2,
    int BN2) {
  pdl_wait();
  pdl_launch_dependents();  // dependents wait for this grid's completion themselves
  small_permutation(idx, w, T, E, k, BN, offsets, gather, row_of, roww, table, table2, BN2);
}

}  // namespace

cudaError_t launch_small_permutation(const int32_t* idx, const float* w, int T, int E, int k,
                                     const SmallPermOut& p, cudaStream_t s) {
  if (T == 0 || T > kSmallT) return cudaErrorInvalidValue;
  return launch_pdl(small_permutation_kernel, dim3(1), dim3(kSmallThreads), 0, s, idx, w, T, E,
                    k, p.BN, p.offsets, p.gather, p.row_of, p.roww, p.table, p.table2, p.BN2);
}

cudaError_t launch_perm_count(const int32_t* idx, int T, int E, int k, int32_t* blockcnt,
                              cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(perm_count_kernel, dim3((T + kPermTokBlock - 1) / kPermTokBlock), dim3(256),
                    0, s, idx, T, E, k, blockcnt);
}

cudaError_t launch_perm_scan(int32_t* blockcnt, int T, int E, int k, int32_t* offsets,
                             int32_t* table, int BN, cudaStream_t s) {
  return launch_pdl(perm_scan_kernel, dim3(1), dim3(1024), 0, s, blockcnt, T, E, k, offsets, table,
                    BN);
}

cudaError_t launch_perm_scatter(const int32_t* idx, const float* w, const int32_t* blockbase,
                                int T, int E, int k, int32_t* gather, int32_t* row_of,
                                float* roww, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(perm_scatter_kernel, dim3((T + kPermTokBlock - 1) / kPermTokBlock), dim3(256),
                    0, s, idx, w, blockbase, T, E, k, gather, row_of, roww);
}

cudaError_t launch_scatter_rows(const uint16_t* x, const int32_t* row_of, int T, int H, int k,
                                bool to_fp16, uint16_t* x_perm, float* zero_out, size_t zero_n,
                                cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (k < 0 || k > kMaxTopK) return cudaErrorInvalidValue;
  // column segments per row: at least 32 chunks each, about 1216 warps in all
  const int chunks = H / 8;
  int segs = 1;
  while (segs < 16 && static_cast<long>(T) * segs < 152 * 8 && chunks % (segs * 2 * 32) == 0)
    segs *= 2;
  const long items = static_cast<long>(T) * segs;
  const int blocks = static_cast<int>(std::min<long>((items + 7) / 8, 152 * 8));
  float4* z4 = reinterpret_cast<float4*>(zero_out);
  const size_t n4 = zero_n / 4;
  if (to_fp16)
    return launch_pdl(scatter_rows_kernel<true>, dim3(blocks), dim3(256), 0, s, x, row_of, T, H, k,
                      segs, x_perm, z4, n4);
  return launch_pdl(scatter_rows_kernel<false>, dim3(blocks), dim3(256), 0, s, x, row_of, T, H, k,
                    segs, x_perm, z4, n4);
}

cudaError_t launch_split_rows_e4m3(const uint16_t* x, const int32_t* row_of, int T, int H, int k,
                                   uint8_t* x8, float* xinv, float* zero_out, size_t zero_n,
                                   cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (k > kMaxTopK || H % 8 != 0) return cudaErrorInvalidValue;
  const int blocks = std::min(T, 1024);
  float4* z4 = reinterpret_cast<float4*>(zero_out);
  return launch_pdl(split_rows_e4m3_kernel, dim3(blocks), dim3(kSplitThreads), 0, s, x, row_of, T,
                    H, k, x8, xinv, z4, zero_out ? zero_n / 4 : 0);
}

cudaError_t launch_table_from_offsets(const int32_t* offsets, int E, int rows, int capacity,
                                      int32_t* table, int BN, cudaStream_t s) {
  return launch_pdl(table_from_offsets_kernel, dim3(1), dim3(1024), 0, s, offsets, E, rows,
                    capacity, table, BN);
}


namespace {

__global__ void __launch_bounds__(256) dense_rows_kernel(int T, int BN, int32_t* __restrict__ gather,
                                                         float* __restrict__ roww,
                                                         int32_t* __restrict__ table) {
  pdl_wait();
  pdl_launch_dependents();  // dependents wait for this grid's completion themselves
  const int n = (T + BN - 1) / BN;
  TileEntry* ent = reinterpret_cast<TileEntry*>(reinterpret_cast<char*>(table) + kTableHeaderBytes);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T || i < n; i += gridDim.x * blockDim.x) {
    if (i < T) {
      gather[i] = i;
      roww[i] = 1.0f;
    }
    if (i < n) {
      TileEntry te;
      te.group = 0;
      te.row0 = i * BN;
      te.nrows = min(BN, T - i * BN);
      te.ntiles = n;
      ent[i] = te;
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) table[0] = n;
}

}  // namespace

cudaError_t launch_dense_rows(int T, int BN, int32_t* gather, float* roww, int32_t* table,
                              cudaStream_t s) {
  const int blocks = min((T + 255) / 256, 152 * 4);
  return launch_pdl(dense_rows_kernel, dim3(blocks > 0 ? blocks : 1), dim3(256), 0, s, T, BN,
                    gather, roww, table);
}

}  // namespace moe
