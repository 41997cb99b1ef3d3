// C ABI of the MoE FFN layer: argument checks, workspace layout, TMA tensor
// maps and the launch sequence of each entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "../../include/moe_ffn.h"
#include "moe_kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr size_t kAlign = 256;
constexpr size_t kHeaderBytes = 256;        // status word + reserved
constexpr size_t kRouteDoneOffset = 64;     // header: CTAs of the top-k kernel done (zero between calls)
constexpr int kRouterTcMinTokens = 256;     // tensor-core router from this many tokens
constexpr int kGatherFromXTokens = 8;       // bf16 gate/up gathers its token rows from x up to this
constexpr int kFusedPermTokens = 16;        // the top-k kernel's last CTA permutes up to this
constexpr int kTmGatherMinTokens = 512;     // token-major gate/up copies its token rows from x from here

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t z, idx, w, blockcnt, offsets, table, table2, gather, row_of, roww, x_perm, xinv, h0, h1,
      hinv, y_perm;
  size_t partial, counters;
  size_t partial_units;  // K-split units the partial buffer holds (0: no split possible)
  size_t ready;          // one-launch decode FFN: counters per entry, then finished CTAs
  int n_ready;           // entries the ready counters cover (0: no one-launch FFN)
  size_t total;
};

int rows_of(const moe_dims& d) { return (d.top_k + 1) * d.T; }

// Token-major grouped GEMMs (tokens as M) serve 128-token tiles.
bool token_major(const moe_dims& d);

int pick_bn(int T) {
  if (T <= 16) return 16;
  if (T <= 32) return 32;
  if (T <= 64) return 64;
  return 128;
}

// Int4 weights up to kInt4GemvMaxTokens tokens, in the shapes the CUDA-core
// kernels take: gate/up and down as GEMVs with 8-bit integer dot products
// (entries of at most kGemvMaxRows rows).  Measured against the 8-bit
// tcgen05 kernels (decode shapes, full layer): 1 token 44.2 vs 64.8 us, 8
// tokens 192.2 vs 206.1, 32 tokens 475.2 vs 516.5, 64 tokens 751.6 vs 730.5.
constexpr int kInt4GemvMaxTokens = 32;

bool int4_gemv(const moe_dims& d) {
  return d.fmt == MOE_W_INT4_G32 && d.T <= kInt4GemvMaxTokens && d.top_k > 0 &&
         int4_gemv_shape_ok(d.H, d.I);
}

// Other Int4 shapes up to 64 tokens: gate/up and down both on 8-bit
// tensor-core operands (gate/up entries of at most kF8MaxRows rows, down
// entries of at most kF8DownMaxRows rows in a table of their own).
bool int4_f8(const moe_dims& d) {
  return d.fmt == MOE_W_INT4_G32 && d.T <= 64 && d.top_k > 0 && d.I <= 4096 && !int4_gemv(d);
}

// Rows per tile-table entry of the fused layer.
int table_bn(const moe_dims& d) {
  return int4_gemv(d) ? kGemvMaxRows : int4_f8(d) ? kF8MaxRows : pick_bn(d.T);
}

size_t table_bytes(const moe_dims& d) {
  // every group contributes at most ceil(cnt / BN) entries with BN >= 5 (the
  // 8-bit down path's entries), so the sum is bounded by (E + 1) + rows / 4
  const size_t entries = static_cast<size_t>(d.E + 1) + (rows_of(d) + 3) / 4;
  return kTableHeaderBytes + entries * sizeof(TileEntry);
}

constexpr int kMaxSplit = 8;
constexpr int kSplitTileLimit = 1024;  // tile counts from which no split is considered

// Upper bound on the tile-table entries of a layer call: at most one entry
// per row and per (group, BN rows).
int entries_bound(const moe_dims& d) {
  const int rows = rows_of(d);
  const int BN = pick_bn(d.T);
  return std::min((d.E + 1) + (rows + BN - 1) / BN, rows);
}

// The fused bf16 layer call runs gate/up and down as one persistent launch
// (decode_ffn_kernel) for weights-as-M tiles up to this many tokens.
constexpr int kOneLaunchFfnMaxTokens = 64;

bool one_launch_ffn(const moe_dims& d) {
  return d.fmt == MOE_W_BF16 && d.top_k > 0 && d.T <= kOneLaunchFfnMaxTokens &&
         pick_bn(d.T) <= 64 && d.I % 128 == 0 && d.H % 256 == 0 &&
         !(d.flags & MOE_FLAG_DETERMINISTIC);
}

// Upper bound on the gate/up tiles of the weight-rows-as-M kernels: at most
// one entry per row and per (group, BN rows).
int gateup_tiles_bound(const moe_dims& d) {
  const int rows = rows_of(d);
  const int BN = pick_bn(d.T);
  // the dense FFN (top_k == 0) is exactly one group of rows
  const int entries = d.top_k == 0 ? (rows + BN - 1) / BN
                                   : std::min((d.E + 1) + (rows + BN - 1) / BN, rows);
  return entries * ((d.I + 127) / 128);
}

// Units per tile along K: enough units for every SM and a last wave at
// least half full; 1 when the tiles alone fill several waves.
int split_for(long tiles, int KB, int nsm) {
  if (tiles <= 0 || tiles >= 4L * nsm) return 1;
  for (int S = 1; S <= kMaxSplit && KB / S >= 4; ++S) {
    const long units = tiles * S;
    if (units < nsm) continue;
    const long full = units / nsm, rem = units % nsm;
    if (rem == 0 || 2 * rem >= nsm || full >= 4) return S;
  }
  return 1;
}

// Units per down tile along I in the one-launch decode FFN: down units add
// into out atomically, so a split costs only atomics; enough units that the
// queue ends with small ones on every SM (about 24 per SM: measured at 8
// tokens, 4 parts instead of 1 took the layer from 354.5 to 346.6 us), at
// least two 64-wide k-steps per unit.
int down_split_for(long tiles, int KB, int nsm) {
  int S = 1;
  while (S < kMaxSplit && tiles * S < 24L * nsm && KB / (S + 1) >= 2) ++S;
  return S;
}

bool token_major(const moe_dims& d) {
  return d.fmt == MOE_W_BF16 && pick_bn(d.T) == 128 && d.I % 128 == 0 && d.H % 256 == 0;
}

Layout layout_of(const moe_dims& d) {
  Layout L{};
  const size_t T = d.T, E = d.E, k = d.top_k, H = d.H, I = d.I, rows = rows_of(d);
  const size_t nblk = (T + kPermTokBlock - 1) / kPermTokBlock;
  size_t o = kHeaderBytes;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  // logits [T][E], or below the tensor-core router's size the partial
  // logits of every reduction slice [slices][T][E]
  L.z = take((d.T < kRouterTcMinTokens ? static_cast<size_t>(router_slices(d.H)) : 1) * T * E * 4);
  L.idx = take(T * k * 4);
  L.w = take(T * k * 4);
  L.blockcnt = take(nblk * E * 4);
  L.offsets = take((E + 2) * 4);
  L.table = take(table_bytes(d));
  L.table2 = take(int4_f8(d) ? table_bytes(d) : 0);  // down entries of the 8-bit path
  L.gather = take(rows * 4);
  L.row_of = take(T * k * 4);
  L.roww = take(rows * 4);
  L.x_perm = take(rows * H * 2);  // Int4 up to 64 tokens: the two e4m3 planes of each row
  L.xinv = take(int4_f8(d) ? rows * 4 : 0);
  L.h0 = take(rows * I * (int4_f8(d) ? 3 : 2));  // 8-bit path: three e4m3 planes of h
  L.h1 = take(d.fmt == MOE_W_BF16 ? rows * I * 2 : 0);
  // 8-bit path: 1 / sigma per row and group of h; CUDA-core path: sigma and
  // 8 sum q per row and group of h
  L.hinv = take(int4_f8(d) ? rows * (I / 32) * 4 : int4_gemv(d) ? rows * (I / 32) * 8 : 0);
  L.y_perm = take((d.flags & MOE_FLAG_DETERMINISTIC) ? rows * H * 4 : 0);
  const int tiles = gateup_tiles_bound(d);
  L.partial_units = tiles < kSplitTileLimit ? static_cast<size_t>(tiles) * kMaxSplit : 0;
  L.partial = take(L.partial_units * 2 * pick_bn(d.T) * 128 * 4);
  L.counters = take(L.partial_units ? static_cast<size_t>(tiles) * 4 : 0);
  L.n_ready = one_launch_ffn(d) ? entries_bound(d) : 0;
  L.ready = take(L.n_ready ? static_cast<size_t>(L.n_ready + 2) * 4 : 0);
  L.total = o;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_dims(const moe_dims* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->T < 0 || d->H <= 0 || d->E <= 0 || d->I <= 0 || d->I_shared <= 0 || d->top_k <= 0)
    return MOE_ERR_INVALID_ARG;
  if (d->fmt != MOE_W_BF16 && d->fmt != MOE_W_INT4_G32) return MOE_ERR_UNSUPPORTED;
  if (d->flags & ~(MOE_FLAG_DETERMINISTIC | MOE_FLAG_ACCUMULATE)) return MOE_ERR_INVALID_ARG;
  if (d->H % 128 != 0 || d->H > 12288) return MOE_ERR_UNSUPPORTED;
  if (d->I % 64 != 0 || d->I_shared != d->I) return MOE_ERR_UNSUPPORTED;
  if (d->E > kMaxE || d->top_k > kMaxTopK || d->top_k > d->E) return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d->T) * (d->top_k + 1) > (1 << 30)) return MOE_ERR_UNSUPPORTED;
  // Int4: a raw stage covers 256 reduction elements and the scale rows
  // (K/32 bf16) must be a whole number of 16-byte TMA strides
  if (d->fmt == MOE_W_INT4_G32 && (d->H % 256 != 0 || d->I % 256 != 0)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status check_device() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// ------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// K-major operand of 16-bit elements [d2][d1][d0] (d0 = reduction, innermost),
// box {64, box_rows, 1}, 128-byte swizzle, zero fill out of bounds.
bool encode_kmajor(CUtensorMap* m, const void* base, bool bf16, uint64_t d0, uint64_t d1,
                   uint64_t d2, uint32_t box_rows) {
  const EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  const cuuint32_t rank = d2 > 1 ? 3 : 2;
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, rank,
            const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Weight stacks are always addressed as 3-D maps (a 2-D map ignores the third
// coordinate, so the shared expert's leading dimension of 1 is fine).
bool encode_weights(CUtensorMap* m, const void* base, bool bf16, uint64_t K, uint64_t N,
                    uint64_t n_experts, uint32_t max_box_rows = 128) {
  const uint32_t box_rows = N < max_box_rows ? static_cast<uint32_t>(N) : max_box_rows;
  const EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {K, N, n_experts};
  const cuuint64_t strides[2] = {K * 2, K * N * 2};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
            const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Codes of an Int4 stack [n][N][K/2] bytes: box {128 bytes, 128 rows, 1},
// 128-byte swizzle (the dequantisers read 16-byte chunks conflict-free).
bool encode_codes(CUtensorMap* m, const void* base, uint64_t K, uint64_t N, uint64_t n_experts) {
  const EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {K / 2, N, n_experts};
  const cuuint64_t strides[2] = {K / 2, K / 2 * N};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scales of an Int4 stack [n][N][K/32] bf16: box {8 groups, 128 rows, 1}
// (256 reduction elements), no swizzle.
bool encode_scales(CUtensorMap* m, const void* base, uint64_t K, uint64_t N, uint64_t n_experts) {
  const EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {K / 32, N, n_experts};
  const cuuint64_t strides[2] = {K / 32 * 2, K / 32 * 2 * N};
  const cuuint32_t box[3] = {8, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// e4m3 activation planes, `plane_rows` rows of K bytes (row P r + p: plane p
// of permuted row r): box {128 bytes, 16 rows}, 128-byte swizzle.
bool encode_e4m3_planes(CUtensorMap* m, const void* base, uint64_t K, uint64_t plane_rows) {
  const EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {K, plane_rows};
  const cuuint64_t strides[1] = {K};
  const cuuint32_t box[2] = {128, 16};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool weights_ok(const moe_weights* w, int fmt) {
  if (!w || !w->gate || !w->up || !w->down) return false;
  if (!aligned16(w->gate) || !aligned16(w->up) || !aligned16(w->down)) return false;
  if (fmt == MOE_W_INT4_G32) {
    if (!w->gate_scale || !w->up_scale || !w->down_scale) return false;
    if (!aligned16(w->gate_scale) || !aligned16(w->up_scale) || !aligned16(w->down_scale))
      return false;
  }
  return true;
}

struct Ws {
  char* base;
  Layout L;
  int* status() const { return reinterpret_cast<int*>(base); }
  int* route_done() const { return reinterpret_cast<int*>(base + kRouteDoneOffset); }
  template <typename T>
  T* at(size_t off) const {
    return reinterpret_cast<T*>(base + off);
  }
};

moe_status check_ws(const moe_dims& d, void* ws, size_t ws_bytes, Ws* out) {
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  out->L = layout_of(d);
  if (ws_bytes < out->L.total) return MOE_ERR_WORKSPACE;
  out->base = static_cast<char*>(ws);
  return MOE_OK;
}

// ------------------------------------------------------------ stages

// Router logits and top-k.  From kRouterTcMinTokens tokens the logits come
// from the tensor cores (bias in the epilogue) and a warp per token selects;
// below, partial logits per reduction slice spread the router matrix over
// all SMs and a warp per token adds the slices, the bias and selects.
// With zero_out, the router's kernels also clear out [T][H]; with perm
// (T <= kSmallT) the top-k kernel's last CTA also runs the permutation.
moe_status run_router(const moe_dims& d, const void* x, const void* w_router, const float* b,
                      int32_t* idx, float* w, const Ws& ws, cudaStream_t s,
                      float* zero_out = nullptr, const SmallPermOut* perm = nullptr) {
  float* z = ws.at<float>(ws.L.z);
  const size_t zero_n = zero_out ? static_cast<size_t>(d.T) * d.H : 0;
  if (d.T < kRouterTcMinTokens) {
    if (launch_router_partials(static_cast<const uint16_t*>(x),
                               static_cast<const uint16_t*>(w_router), z, d.T, d.H, d.E,
                               zero_out, zero_n, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    return from_cuda(
        launch_router_reduce_topk(z, b, d.T, d.H, d.E, d.top_k, idx, w, nullptr, perm, s));
  }
  cudaError_t e;
  {
    DownLaunch L{};
    if (!encode_weights(&L.tm_a, w_router, true, d.H, d.E, 1) ||
        !encode_kmajor(&L.tm_b0, x, true, d.H, d.T, 1, 16))
      return MOE_ERR_CUDA;
    L.tm_a_shared = L.tm_a;
    L.tm_b1 = L.tm_b0;
    L.table = nullptr;
    L.dense_rows = d.T;
    L.BN = 128;
    L.nb = 1;
    L.K = d.H;
    L.N_out = d.E;
    L.mblocks = (d.E + 127) / 128;
    L.E = -1;
    L.a_rows = d.E < 128 ? d.E : 128;
    L.total_rows = d.T;
    L.out_rows = d.T;
    L.bf16 = true;
    L.epilogue = kEpiRouter;
    L.ksplit = 1;
    L.bias = b;
    L.out = z;
    L.status = ws.status();
    L.budget_ns = kWaitBudgetNs;
    const int tiles = ((d.T + 127) / 128) * L.mblocks;
    L.grid = tiles < sm_count() ? tiles : sm_count();
    e = launch_down(L, s);
  }
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return from_cuda(launch_topk(z, d.T, d.E, d.top_k, idx, w, s, zero_out, zero_n));
}

// materialise: also write x_perm (and clear zero_out) with the gather kernel;
// the fused bf16 path leaves it out, its GEMMs read the rows from x.
moe_status run_permute(const moe_dims& d, const int32_t* idx, const float* w, const void* x,
                       int32_t* offsets, int32_t* gather, int32_t* row_of, float* roww,
                       void* x_perm, int32_t* table, const Ws& ws, cudaStream_t s,
                       float* zero_out = nullptr, bool materialise = true) {
  cudaError_t e;
  if (d.T <= kSmallT) {
    // the one-CTA permutation the fused call runs at these sizes
    const SmallPermOut p{nullptr, pick_bn(d.T), offsets, gather, row_of, roww, table, nullptr, 0};
    e = launch_small_permutation(idx, w, d.T, d.E, d.top_k, p, s);
  } else {
    int32_t* blockcnt = ws.at<int32_t>(ws.L.blockcnt);
    e = launch_perm_count(idx, d.T, d.E, d.top_k, blockcnt, s);
    if (e == cudaSuccess)
      e = launch_perm_scan(blockcnt, d.T, d.E, d.top_k, offsets, table, pick_bn(d.T), s);
    if (e == cudaSuccess)
      e = launch_perm_scatter(idx, w, blockcnt, d.T, d.E, d.top_k, gather, row_of, roww, s);
  }
  if (e == cudaSuccess && materialise)
    e = launch_scatter_rows(static_cast<const uint16_t*>(x), row_of, d.T, d.H, d.top_k,
                            d.fmt == MOE_W_INT4_G32, static_cast<uint16_t*>(x_perm), zero_out,
                            zero_out ? static_cast<size_t>(d.T) * d.H : 0, s);
  return from_cuda(e);
}

// Under stream capture the records become event nodes of the graph, so that
// every replay times its own stages.
void record(const moe_stage_events* ev, int i, cudaStream_t s) {
  if (!ev || !ev->ev[i]) return;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cap);
  cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev->ev[i]), s,
                           cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal
                                                                : cudaEventRecordDefault);
}

// Grouped gate/up + down over the permuted rows described by `table`.
// Token rows: x_perm [rows][H] (xrows null), or with xrows (bf16 weights,
// the weights-as-M kernels) the gate/up GEMM reads row r as x[xrows[r]]
// straight from x = `x_perm` [T][H].
moe_status run_experts(const moe_dims& d, const void* x_perm, const int32_t* table,
                       const moe_weights* ex, const moe_weights* sh, int epilogue,
                       const int32_t* gather, const float* roww, float* out, const Ws& ws,
                       cudaStream_t s, const moe_stage_events* ev = nullptr,
                       const int32_t* xrows = nullptr, float* zero_out = nullptr,
                       const float* xinv = nullptr, const int32_t* down_table = nullptr,
                       const void* x_shared_first = nullptr) {
  const int rows = rows_of(d);
  const int nsm = sm_count();
  if (d.fmt == MOE_W_INT4_G32 && xrows && int4_gemv(d)) {
    // CUDA-core GEMVs: gate/up quantises the rows x[xrows[r]] itself and
    // writes h as 16-bit planes, down reads them through the same table
    Int4GemvLaunch G{};
    G.table = table;
    G.E = d.E;
    G.total_rows = rows;
    G.out_rows = d.T;
    G.x = static_cast<const uint16_t*>(x_perm);
    G.xrows = xrows;
    G.hq = ws.at<uint8_t>(ws.L.h0);
    G.hs = ws.at<float>(ws.L.hinv);
    G.hc = reinterpret_cast<int32_t*>(G.hs + static_cast<size_t>(rows) * (d.I / 32));
    Int4GemvLaunch D = G;
    G.K = d.H;
    G.N_out = d.I;
    G.codes[0] = ex->gate;
    G.codes[1] = ex->up;
    G.scale[0] = ex->gate_scale;
    G.scale[1] = ex->up_scale;
    G.scodes[0] = sh->gate;
    G.scodes[1] = sh->up;
    G.sscale[0] = sh->gate_scale;
    G.sscale[1] = sh->up_scale;
    const long entries = std::min<long>((d.E + 1) + (rows + kGemvMaxRows - 1) / kGemvMaxRows, rows);
    G.grid = static_cast<int>(std::min<long>(entries * (d.I / 32), 2L * nsm));
    record(ev, 2, s);
    if (launch_int4_gemv_gateup(G, s) != cudaSuccess) return MOE_ERR_CUDA;
    record(ev, 3, s);
    D.epilogue = epilogue;
    D.K = d.I;
    D.N_out = d.H;
    D.codes[0] = D.codes[1] = ex->down;
    D.scale[0] = D.scale[1] = ex->down_scale;
    D.scodes[0] = D.scodes[1] = sh->down;
    D.sscale[0] = D.sscale[1] = sh->down_scale;
    D.gather = gather;
    D.roww = roww;
    D.out = out;
    D.grid = static_cast<int>(std::min<long>(entries * (d.H / 128), 2L * nsm));
    const cudaError_t e = launch_int4_gemv_down(D, s);
    record(ev, 4, s);
    return from_cuda(e);
  }
  if (d.fmt == MOE_W_INT4_G32 && xinv && down_table) {
    // 8-bit operands: x_perm holds the e4m3 planes of x; gate/up writes h as
    // three planes, down reads them through its own table
    uint8_t* h8 = ws.at<uint8_t>(ws.L.h0);
    float* hinv = ws.at<float>(ws.L.hinv);
    Int4F8Launch G{};
    if (!encode_codes(&G.tm_c[0], ex->gate, d.H, d.I, d.E) ||
        !encode_codes(&G.tm_c[1], ex->up, d.H, d.I, d.E) ||
        !encode_codes(&G.tm_sc[0], sh->gate, d.H, d.I, 1) ||
        !encode_codes(&G.tm_sc[1], sh->up, d.H, d.I, 1) ||
        !encode_e4m3_planes(&G.tm_b, x_perm, d.H, 2 * static_cast<uint64_t>(rows)))
      return MOE_ERR_CUDA;
    G.table = table;
    G.na = 2;
    G.epilogue = kEpiStoreRows;
    G.K = d.H;
    G.N_out = d.I;
    G.E = d.E;
    G.total_rows = rows;
    G.out_rows = d.T;
    G.scale[0] = ex->gate_scale;
    G.scale[1] = ex->up_scale;
    G.sscale[0] = sh->gate_scale;
    G.sscale[1] = sh->up_scale;
    G.binv = xinv;
    G.h8 = h8;
    G.hinv = hinv;
    G.status = ws.status();
    G.budget_ns = kWaitBudgetNs;
    const int gentries = (d.E + 1) + (rows + kF8MaxRows - 1) / kF8MaxRows;
    const int gtiles = gentries * (d.I / 128);
    G.grid = gtiles < nsm ? gtiles : nsm;
    record(ev, 2, s);
    if (launch_int4_f8_gemm(G, s) != cudaSuccess) return MOE_ERR_CUDA;
    record(ev, 3, s);
    Int4F8Launch D{};
    if (!encode_codes(&D.tm_c[0], ex->down, d.I, d.H, d.E) ||
        !encode_codes(&D.tm_sc[0], sh->down, d.I, d.H, 1) ||
        !encode_e4m3_planes(&D.tm_b, h8, d.I, 3 * static_cast<uint64_t>(rows)))
      return MOE_ERR_CUDA;
    D.tm_c[1] = D.tm_c[0];
    D.tm_sc[1] = D.tm_sc[0];
    D.table = down_table;
    // the scatter-add down runs tiles of two 128-row blocks (H % 256 == 0 for Int4)
    const bool pair = epilogue == kEpiScatterAdd;
    D.na = pair ? 2 : 1;
    D.epilogue = epilogue;
    D.K = d.I;
    D.N_out = d.H;
    D.E = d.E;
    D.total_rows = rows;
    D.out_rows = d.T;
    D.scale[0] = D.scale[1] = ex->down_scale;
    D.sscale[0] = D.sscale[1] = sh->down_scale;
    D.binv = hinv;
    D.gather = gather;
    D.roww = roww;
    D.out = out;
    D.status = ws.status();
    D.budget_ns = kWaitBudgetNs;
    const int dentries = (d.E + 1) + (rows + kF8DownMaxRows - 1) / kF8DownMaxRows;
    const int dtiles = dentries * (d.H / (pair ? 256 : 128));
    D.grid = dtiles < nsm ? dtiles : nsm;
    const cudaError_t e = launch_int4_f8_gemm(D, s);
    record(ev, 4, s);
    return from_cuda(e);
  }
  const int BN = pick_bn(d.T);
  const int max_entries = (d.E + 1) + (rows + BN - 1) / BN;
  if (d.fmt == MOE_W_INT4_G32) {
    Int4Launch G{};
    if (!encode_codes(&G.tm_c[0], ex->gate, d.H, d.I, d.E) ||
        !encode_codes(&G.tm_c[1], ex->up, d.H, d.I, d.E) ||
        !encode_scales(&G.tm_s[0], ex->gate_scale, d.H, d.I, d.E) ||
        !encode_scales(&G.tm_s[1], ex->up_scale, d.H, d.I, d.E) ||
        !encode_codes(&G.tm_sc[0], sh->gate, d.H, d.I, 1) ||
        !encode_codes(&G.tm_sc[1], sh->up, d.H, d.I, 1) ||
        !encode_scales(&G.tm_ss[0], sh->gate_scale, d.H, d.I, 1) ||
        !encode_scales(&G.tm_ss[1], sh->up_scale, d.H, d.I, 1) ||
        !encode_kmajor(&G.tm_b, x_perm, false, d.H, rows, 1, 16))
      return MOE_ERR_CUDA;
    G.table = table;
    G.BN = BN;
    G.na = 2;
    G.K = d.H;
    G.N_out = d.I;
    G.mblocks = d.I / 128;
    G.E = d.E;
    G.total_rows = rows;
    G.out_rows = d.T;
    G.epilogue = kEpiStoreRows;
    G.h = ws.at<void>(ws.L.h0);
    G.status = ws.status();
    G.budget_ns = kWaitBudgetNs;
    G.grid = max_entries * G.mblocks < nsm ? max_entries * G.mblocks : nsm;
    record(ev, 2, s);
    if (launch_int4_gemm(G, s) != cudaSuccess) return MOE_ERR_CUDA;
    record(ev, 3, s);
    Int4Launch D{};
    if (!encode_codes(&D.tm_c[0], ex->down, d.I, d.H, d.E) ||
        !encode_scales(&D.tm_s[0], ex->down_scale, d.I, d.H, d.E) ||
        !encode_codes(&D.tm_sc[0], sh->down, d.I, d.H, 1) ||
        !encode_scales(&D.tm_ss[0], sh->down_scale, d.I, d.H, 1) ||
        !encode_kmajor(&D.tm_b, G.h, false, d.I, rows, 1, 16))
      return MOE_ERR_CUDA;
    D.tm_c[1] = D.tm_c[0];
    D.tm_s[1] = D.tm_s[0];
    D.tm_sc[1] = D.tm_sc[0];
    D.tm_ss[1] = D.tm_ss[0];
    D.table = table;
    D.BN = BN;
    // the scatter-add down runs tiles of two 128-row blocks (H % 256 == 0 for Int4)
    const bool pair = epilogue == kEpiScatterAdd;
    D.na = pair ? 2 : 1;
    D.K = d.I;
    D.N_out = d.H;
    D.mblocks = d.H / (pair ? 256 : 128);
    D.E = d.E;
    D.total_rows = rows;
    D.out_rows = d.T;
    D.epilogue = epilogue;
    D.gather = gather;
    D.roww = roww;
    D.out = out;
    D.status = ws.status();
    D.budget_ns = kWaitBudgetNs;
    D.grid = max_entries * D.mblocks < nsm ? max_entries * D.mblocks : nsm;
    const cudaError_t e = launch_int4_gemm(D, s);
    record(ev, 4, s);
    return from_cuda(e);
  }

  if (token_major(d)) {
    // token-major kernels: tiles of up to 128 rows of one group
    TmLaunch G{};
    // with xrows the producer warp copies the token rows from x itself
    if (!encode_kmajor(&G.tm_a[0], x_perm, true, d.H, xrows ? d.T : rows, 1, 128) ||
        !encode_weights(&G.tm_b[0], ex->gate, true, d.H, d.I, d.E, 128) ||
        !encode_weights(&G.tm_b[1], ex->up, true, d.H, d.I, d.E, 128) ||
        !encode_weights(&G.tm_sb[0], sh->gate, true, d.H, d.I, 1, 128) ||
        !encode_weights(&G.tm_sb[1], sh->up, true, d.H, d.I, 1, 128))
      return MOE_ERR_CUDA;
    G.tm_a[1] = G.tm_a[0];
    G.table = table;
    G.arows = xrows;
    G.xsrc = x_perm;
    G.xpitch = d.H;
    G.zero_out = zero_out;
    G.zero_n = zero_out ? static_cast<size_t>(d.T) * d.H : 0;
    G.gateup = true;
    G.K = d.H;
    G.N_out = d.I;
    G.nblocks = d.I / 128;
    G.E = d.E;
    G.total_rows = rows;
    G.out_rows = d.T;
    G.epilogue = kEpiStoreRows;
    G.h0 = ws.at<void>(ws.L.h0);
    G.h1 = ws.at<void>(ws.L.h1);
    G.status = ws.status();
    G.budget_ns = kWaitBudgetNs;
    G.grid = max_entries * G.nblocks < nsm ? max_entries * G.nblocks : nsm;
    record(ev, 2, s);
    if (launch_tm_gemm(G, s) != cudaSuccess) return MOE_ERR_CUDA;
    record(ev, 3, s);
    TmLaunch D{};
    if (!encode_kmajor(&D.tm_a[0], G.h0, true, d.I, rows, 1, 128) ||
        !encode_kmajor(&D.tm_a[1], G.h1, true, d.I, rows, 1, 128) ||
        !encode_weights(&D.tm_b[0], ex->down, true, d.I, d.H, d.E, 256) ||
        !encode_weights(&D.tm_sb[0], sh->down, true, d.I, d.H, 1, 256))
      return MOE_ERR_CUDA;
    D.tm_b[1] = D.tm_b[0];
    D.tm_sb[1] = D.tm_sb[0];
    D.table = table;
    D.gateup = false;
    D.K = d.I;
    D.N_out = d.H;
    D.nblocks = d.H / 256;
    D.E = d.E;
    D.total_rows = rows;
    D.out_rows = d.T;
    D.epilogue = epilogue;
    D.gather = gather;
    D.roww = roww;
    D.out = out;
    D.status = ws.status();
    D.budget_ns = kWaitBudgetNs;
    D.grid = max_entries * D.nblocks < nsm ? max_entries * D.nblocks : nsm;
    const cudaError_t e = launch_tm_gemm(D, s);
    record(ev, 4, s);
    return from_cuda(e);
  }

  GateUpLaunch G{};
  const bool bf16 = true;
  if (!encode_weights(&G.tm_gate, ex->gate, bf16, d.H, d.I, d.E) ||
      !encode_weights(&G.tm_up, ex->up, bf16, d.H, d.I, d.E) ||
      !encode_weights(&G.tm_sgate, sh->gate, bf16, d.H, d.I, 1) ||
      !encode_weights(&G.tm_sup, sh->up, bf16, d.H, d.I, 1) ||
      !(xrows ? encode_kmajor(&G.tm_x, x_perm, bf16, d.H, d.T, 1, 1)
              : encode_kmajor(&G.tm_x, x_perm, bf16, d.H, rows, 1, 16)))
    return MOE_ERR_CUDA;
  G.table = table;
  G.xrows = xrows;
  G.BN = BN;
  // fused layer: the shared expert's tiles (rows = the tokens in order) run
  // before the kernel waits for the routing, reading x directly
  if (x_shared_first && d.top_k > 0) {
    if (!encode_kmajor(&G.tm_xs, x_shared_first, bf16, d.H, d.T, 1, 16)) return MOE_ERR_CUDA;
    G.n_sh = (d.T + BN - 1) / BN;
    G.T = d.T;
    G.sh_row0 = d.top_k * d.T;
  } else {
    G.tm_xs = G.tm_x;
    G.n_sh = 0;
  }
  G.K = d.H;
  G.I = d.I;
  G.E = d.E;
  G.a_rows = d.I < 128 ? d.I : 128;
  G.total_rows = rows;
  G.bf16 = bf16;
  G.h0 = ws.at<void>(ws.L.h0);
  G.h1 = ws.at<void>(ws.L.h1);
  G.status = ws.status();
  G.budget_ns = kWaitBudgetNs;
  {
    const int tiles = gateup_tiles_bound(d);
    int S = split_for(tiles, d.H / 64, nsm);
    if (static_cast<size_t>(tiles) * S > ws.L.partial_units) S = 1;
    G.ksplit = S;
    G.partial = ws.at<float>(ws.L.partial);
    G.counters = ws.at<int>(ws.L.counters);
    const long units = static_cast<long>(tiles) * S;
    G.grid = units < nsm ? static_cast<int>(units) : nsm;
  }
  // the fused layer call: gate/up and down as one persistent launch
  const bool one_launch = x_shared_first && G.n_sh > 0 && epilogue == kEpiScatterAdd &&
                          ws.L.n_ready > 0 && one_launch_ffn(d);
  if (!one_launch) {
    record(ev, 2, s);
    if (launch_gateup(G, s) != cudaSuccess) return MOE_ERR_CUDA;
    record(ev, 3, s);
  }

  DownLaunch D{};
  if (!encode_weights(&D.tm_a, ex->down, bf16, d.I, d.H, d.E) ||
      !encode_weights(&D.tm_a_shared, sh->down, bf16, d.I, d.H, 1) ||
      !encode_kmajor(&D.tm_b0, G.h0, true, d.I, rows, 1, 16) ||
      !encode_kmajor(&D.tm_b1, G.h1, true, d.I, rows, 1, 16))
    return MOE_ERR_CUDA;
  D.table = table;
  D.dense_rows = 0;
  D.BN = BN;
  D.nb = 2;
  D.K = d.I;
  D.N_out = d.H;
  D.mblocks = d.H / 128;
  D.E = d.E;
  D.a_rows = 128;
  D.total_rows = rows;
  D.out_rows = d.T;
  D.bf16 = true;
  D.epilogue = epilogue;
  D.gather = gather;
  D.roww = roww;
  D.bias = nullptr;
  D.out = out;
  D.status = ws.status();
  D.budget_ns = kWaitBudgetNs;
  {
    const int entries = d.top_k == 0 ? (rows + BN - 1) / BN : std::min(max_entries, rows);
    const long tiles = static_cast<long>(entries) * D.mblocks;
    // a split down projection adds its parts atomically (order varies), so
    // not in the deterministic mode
    D.ksplit = (epilogue == kEpiScatterAdd && !(d.flags & MOE_FLAG_DETERMINISTIC))
                   ? split_for(tiles, d.I / 64, nsm) : 1;
    const long units = tiles * D.ksplit;
    D.grid = units < nsm ? static_cast<int>(units) : nsm;
  }
  if (one_launch) {
    FfnLaunch F{};
    F.g = G;
    F.tm_down = D.tm_a;
    F.tm_sdown = D.tm_a_shared;
    F.tm_h0 = D.tm_b0;
    F.tm_h1 = D.tm_b1;
    // down units of 256 output features (two row blocks against one h tile)
    F.ks_d = down_split_for(static_cast<long>(std::min(max_entries, rows)) * (d.H / 256), d.I / 64,
                            nsm);
    F.ready = ws.at<int>(ws.L.ready);
    F.n_ready = ws.L.n_ready;
    F.gather = gather;
    F.roww = roww;
    F.out = out;
    F.out_rows = d.T;
    // one CTA per SM at most: the units wait on one another across CTAs
    const long units = static_cast<long>(ws.L.n_ready) *
                       ((d.I / 128) * G.ksplit + (d.H / 256) * F.ks_d);
    F.grid = units < nsm ? static_cast<int>(units) : nsm;
    // one kernel: the gate/up stage event brackets it, the down stage is empty
    record(ev, 2, s);
    const cudaError_t e = launch_decode_ffn(F, s);
    record(ev, 3, s);
    record(ev, 4, s);
    return from_cuda(e);
  }
  const cudaError_t e = launch_down(D, s);
  record(ev, 4, s);
  return from_cuda(e);
}

moe_status forward_impl(const moe_dims* d, const void* x, const void* w_router,
                        const float* b_router, const moe_weights* experts,
                        const moe_weights* shared, float* out, void* ws, size_t ws_bytes,
                        const moe_stage_events* ev, moe_stream_t stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;  // nothing is read or written
  if (!x || !w_router || !b_router || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if (!weights_ok(experts, d->fmt) || !weights_ok(shared, d->fmt)) return MOE_ERR_INVALID_ARG;
  Ws w;
  if ((st = check_ws(*d, ws, ws_bytes, &w)) != MOE_OK) return st;
  if ((st = check_device()) != MOE_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const Layout& L = w.L;
  int32_t* idx = w.at<int32_t>(L.idx);
  float* wts = w.at<float>(L.w);
  int32_t* gather = w.at<int32_t>(L.gather);
  float* roww = w.at<float>(L.roww);
  int32_t* table = w.at<int32_t>(L.table);
  void* x_perm = w.at<void>(L.x_perm);
  const bool det = (d->flags & MOE_FLAG_DETERMINISTIC) != 0;
  const bool accumulate = (d->flags & MOE_FLAG_ACCUMULATE) != 0;
  // out is cleared (by the router kernels, or for Int4 by the gather that
  // converts x) only when the down epilogue adds into it
  float* zero_out = (det || accumulate) ? nullptr : out;
  // bf16 weights: the gate/up GEMM gathers each token row straight from x,
  // so the permuted copy of x and its kernel drop out -- up to
  // kGatherFromXTokens tokens by TMA tile::gather4 (above that the gathers
  // cost the copy engine more than the copy kernel, measured), and from
  // kTmGatherMinTokens tokens in the token-major kernels by cp.async from a
  // gather warp (measured: -3.1 % per step at 4096 tokens, -0.6 % at 512,
  // +0.8 % at 128).  Int4 needs the fp16 copy in its operand order, or up
  // to 64 tokens the two e4m3 planes of the 8-bit gate/up kernel, except in
  // the CUDA-core kernels, which quantise the rows of x themselves.
  const bool int4 = d->fmt == MOE_W_INT4_G32;
  const bool f8 = int4_f8(*d);
  const bool gemv = int4_gemv(*d);
  float* xinv = f8 ? w.at<float>(L.xinv) : nullptr;
  const bool tm = token_major(*d);
  const bool rows_from_x =
      gemv || (!int4 && (d->T <= kGatherFromXTokens || (tm && d->T >= kTmGatherMinTokens)));
  // who clears out: the gather kernel when it runs, else the token-major
  // gate/up kernel's idle epilogue warps, else the router's kernels
  float* zero_gather = rows_from_x ? nullptr : zero_out;
  float* zero_gemm = rows_from_x && tm ? zero_out : nullptr;
  float* zero_router = rows_from_x && !tm ? zero_out : nullptr;
  // decode sizes: one CTA permutes; up to kFusedPermTokens tokens it is the
  // top-k kernel's last CTA (one launch fewer), above a launch of its own
  // with more threads (measured faster at 64 tokens)
  int32_t* table2 = f8 ? w.at<int32_t>(L.table2) : nullptr;
  const SmallPermOut perm{w.route_done(), table_bn(*d), w.at<int32_t>(L.offsets), gather,
                          w.at<int32_t>(L.row_of), roww, table, table2, kF8DownMaxRows};
  const bool small = d->T <= kSmallT, fused = d->T <= kFusedPermTokens;
  // up to 16 tokens (H <= 4096) one launch routes and permutes (measured at
  // one token: 18 us of routing kernels before)
  const bool one_launch = d->T <= kRouteSmallT && d->H <= 4096;
  record(ev, 0, s);
  if (one_launch) {
    if (launch_route_small(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(w_router),
                           b_router, d->T, d->H, d->E, d->top_k, w.at<float>(L.z), idx, wts, perm,
                           zero_router, zero_router ? static_cast<size_t>(d->T) * d->H : 0,
                           s) != cudaSuccess)
      return MOE_ERR_CUDA;
  } else if ((st = run_router(*d, x, w_router, b_router, idx, wts, w, s, zero_router,
                              fused ? &perm : nullptr)) != MOE_OK) {
    return st;
  }
  record(ev, 1, s);
  if (small) {
    if (!fused && launch_small_permutation(idx, wts, d->T, d->E, d->top_k, perm, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    const size_t zn = zero_gather ? static_cast<size_t>(d->T) * d->H : 0;
    if (f8) {
      if (launch_split_rows_e4m3(static_cast<const uint16_t*>(x), w.at<int32_t>(L.row_of), d->T,
                                 d->H, d->top_k, static_cast<uint8_t*>(x_perm), xinv, zero_gather,
                                 zn, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    } else if (!rows_from_x &&
               launch_scatter_rows(static_cast<const uint16_t*>(x), w.at<int32_t>(L.row_of), d->T,
                                   d->H, d->top_k, int4, static_cast<uint16_t*>(x_perm),
                                   zero_gather, zn, s) != cudaSuccess) {
      return MOE_ERR_CUDA;
    }
  } else {
    if ((st = run_permute(*d, idx, wts, x, w.at<int32_t>(L.offsets), gather,
                          w.at<int32_t>(L.row_of), roww, x_perm, table, w, s, zero_gather,
                          !rows_from_x)) != MOE_OK)
      return st;
  }
  const void* rows_src = rows_from_x ? x : x_perm;
  const int32_t* xrows = rows_from_x ? gather : nullptr;
  if (!det)
    return run_experts(*d, rows_src, table, experts, shared, kEpiScatterAdd, gather, roww, out, w,
                       s, ev, xrows, zero_gemm, xinv, table2, x);
  // deterministic: unweighted rows, then the fixed-order combination
  float* y_perm = w.at<float>(L.y_perm);
  if ((st = run_experts(*d, rows_src, table, experts, shared, kEpiStoreRows, nullptr, nullptr,
                        y_perm, w, s, ev, xrows, zero_gemm, xinv, table2, x)) != MOE_OK)
    return st;
  const cudaError_t e = launch_combine(y_perm, w.at<int32_t>(L.row_of), wts, d->T, d->H,
                                       d->top_k, accumulate, out, s);
  record(ev, 4, s);
  return from_cuda(e);
}

// Dims of the dense FFN as a one-group problem: group 0 = all T rows.
moe_dims dense_dims(const moe_dims& d) {
  moe_dims dd = d;
  dd.E = 1;
  dd.top_k = 0;
  dd.I_shared = d.I;
  dd.flags = d.flags & MOE_FLAG_DETERMINISTIC;
  return dd;
}

moe_status check_dense_dims(const moe_dims* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->T < 0 || d->H <= 0 || d->I <= 0) return MOE_ERR_INVALID_ARG;
  if (d->fmt != MOE_W_BF16 && d->fmt != MOE_W_INT4_G32) return MOE_ERR_UNSUPPORTED;
  if (d->flags & ~(MOE_FLAG_DETERMINISTIC | MOE_FLAG_ACCUMULATE)) return MOE_ERR_INVALID_ARG;
  if (d->H % 128 != 0 || d->H > 12288 || d->I % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (d->fmt == MOE_W_INT4_G32 && (d->H % 256 != 0 || d->I % 256 != 0)) return MOE_ERR_UNSUPPORTED;
  if (d->T > (1 << 30)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_abi_version(void) { return MOE_FFN_ABI_VERSION; }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: null, misaligned or negative argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: shape, format or GPU not supported";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace smaller than moe_workspace_size()";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call failed";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a device-side wait ran out of time";
  }
  return "unknown moe_status";
}

size_t moe_workspace_size(const moe_dims* d) {
  if (check_dims(d) != MOE_OK) return 0;
  return layout_of(*d).total;
}

moe_status moe_router_topk(const moe_dims* d, const void* x, const void* w_router,
                           const float* b_router, int32_t* topk_idx, float* topk_w, void* ws,
                           size_t ws_bytes, moe_stream_t stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;  // nothing is read or written
  if (!x || !w_router || !b_router || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router)) return MOE_ERR_INVALID_ARG;
  Ws w;
  if ((st = check_ws(*d, ws, ws_bytes, &w)) != MOE_OK) return st;
  if ((st = check_device()) != MOE_OK) return st;
  return run_router(*d, x, w_router, b_router, topk_idx, topk_w, w,
                    reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_permute(const moe_dims* d, const int32_t* topk_idx, const void* x,
                       int32_t* offsets, int32_t* gather, int32_t* row_of, void* x_perm, void* ws,
                       size_t ws_bytes, moe_stream_t stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;  // nothing is read or written
  if (!topk_idx || !x || !offsets || !gather || !row_of || !x_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_INVALID_ARG;
  Ws w;
  if ((st = check_ws(*d, ws, ws_bytes, &w)) != MOE_OK) return st;
  if ((st = check_device()) != MOE_OK) return st;
  return run_permute(*d, topk_idx, nullptr, x, offsets, gather, row_of, nullptr, x_perm,
                     w.at<int32_t>(w.L.table), w, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_expert_ffn(const moe_dims* d, const void* x_perm, const int32_t* offsets,
                          const moe_weights* experts, const moe_weights* shared, float* y_perm,
                          void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;  // nothing is read or written
  if (!x_perm || !offsets || !y_perm || !aligned16(x_perm)) return MOE_ERR_INVALID_ARG;
  if (!weights_ok(experts, d->fmt) || !weights_ok(shared, d->fmt)) return MOE_ERR_INVALID_ARG;
  Ws w;
  if ((st = check_ws(*d, ws, ws_bytes, &w)) != MOE_OK) return st;
  if ((st = check_device()) != MOE_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* table = w.at<int32_t>(w.L.table);
  const int capacity =
      static_cast<int>((table_bytes(*d) - kTableHeaderBytes) / sizeof(TileEntry));
  if (launch_table_from_offsets(offsets, d->E, rows_of(*d), capacity, table, pick_bn(d->T), s) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return run_experts(*d, x_perm, table, experts, shared, kEpiStoreRows, nullptr, nullptr, y_perm,
                     w, s);
}

moe_status moe_combine(const moe_dims* d, const float* y_perm, const int32_t* row_of,
                       const float* topk_w, float* out, moe_stream_t stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;  // nothing is read or written
  if (!y_perm || !row_of || !topk_w || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  return from_cuda(launch_combine(y_perm, row_of, topk_w, d->T, d->H, d->top_k,
                                  (d->flags & MOE_FLAG_ACCUMULATE) != 0, out,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_ffn_forward(const moe_dims* d, const void* x, const void* w_router,
                           const float* b_router, const moe_weights* experts,
                           const moe_weights* shared, float* out, void* ws, size_t ws_bytes,
                           moe_stream_t stream) {
  return forward_impl(d, x, w_router, b_router, experts, shared, out, ws, ws_bytes, nullptr,
                      stream);
}

moe_status moe_ffn_forward_timed(const moe_dims* d, const void* x, const void* w_router,
                                 const float* b_router, const moe_weights* experts,
                                 const moe_weights* shared, float* out, void* ws,
                                 size_t ws_bytes, const moe_stage_events* events,
                                 moe_stream_t stream) {
  return forward_impl(d, x, w_router, b_router, experts, shared, out, ws, ws_bytes, events,
                      stream);
}

size_t moe_dense_workspace_size(const moe_dims* d) {
  if (check_dense_dims(d) != MOE_OK) return 0;
  return layout_of(dense_dims(*d)).total;
}

moe_status moe_dense_ffn(const moe_dims* d, const void* x, const moe_weights* weights, float* out,
                         void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status st = check_dense_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;
  if (!x || !out || !aligned16(x) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if (!weights_ok(weights, d->fmt)) return MOE_ERR_INVALID_ARG;
  const moe_dims dd = dense_dims(*d);
  Ws w;
  if ((st = check_ws(dd, ws, ws_bytes, &w)) != MOE_OK) return st;
  if ((st = check_device()) != MOE_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* gather = w.at<int32_t>(w.L.gather);
  float* roww = w.at<float>(w.L.roww);
  int32_t* table = w.at<int32_t>(w.L.table);
  if (launch_dense_rows(d->T, pick_bn(d->T), gather, roww, table, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!(d->flags & MOE_FLAG_ACCUMULATE) &&
      cudaMemsetAsync(out, 0, static_cast<size_t>(d->T) * d->H * sizeof(float), s) != cudaSuccess)
    return MOE_ERR_CUDA;
  const void* rows = x;
  if (d->fmt == MOE_W_INT4_G32) {  // the Int4 GEMMs take fp16 activations
    if (launch_scatter_rows(static_cast<const uint16_t*>(x), nullptr, d->T, d->H, 0, true,
                            w.at<uint16_t>(w.L.x_perm), nullptr, 0, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    rows = w.at<void>(w.L.x_perm);
  }
  // one contribution per output element: the atomic add onto zero (or onto
  // the caller's values) gives the same bits on every run
  return run_experts(dd, rows, table, weights, weights, kEpiScatterAdd, gather, roww, out, w, s);
}

int moe_ffn_one_launch(const moe_dims* d) {
  if (check_dims(d) != MOE_OK) return -1;
  return one_launch_ffn(*d) ? 1 : 0;
}

int moe_ffn_int4_gemv(const moe_dims* d) {
  if (check_dims(d) != MOE_OK) return -1;
  return int4_gemv(*d) ? 1 : 0;
}

moe_status moe_workspace_routing(const moe_dims* d, const void* ws, size_t ws_bytes,
                                 moe_routing_view* view) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (!view) return MOE_ERR_INVALID_ARG;
  *view = moe_routing_view{};
  if (d->T == 0) return MOE_OK;
  Ws w;
  if ((st = check_ws(*d, const_cast<void*>(ws), ws_bytes, &w)) != MOE_OK) return st;
  view->topk_idx = w.at<const int32_t>(w.L.idx);
  view->topk_w = w.at<const float>(w.L.w);
  view->offsets = w.at<const int32_t>(w.L.offsets);
  view->gather = w.at<const int32_t>(w.L.gather);
  view->row_of = w.at<const int32_t>(w.L.row_of);
  return MOE_OK;
}

moe_status moe_tp_slice_weights(const moe_dims* d, int32_t n_experts, int32_t part,
                                int32_t parts, const moe_weights* full, const moe_weights* slice,
                                moe_stream_t stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (n_experts < 1 || parts < 1 || part < 0 || part >= parts) return MOE_ERR_INVALID_ARG;
  if (d->I % parts != 0) return MOE_ERR_UNSUPPORTED;
  const bool int4 = d->fmt == MOE_W_INT4_G32;
  const size_t I = d->I, H = d->H, Is = I / parts, n = n_experts, p = part;
  // each slice must itself be a valid intermediate size
  if (Is % (int4 ? 256 : 64) != 0) return MOE_ERR_UNSUPPORTED;
  if (!weights_ok(full, d->fmt) || !weights_ok(slice, d->fmt)) return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto dst = [](const void* q) { return const_cast<void*>(q); };
  auto src = [](const void* q, size_t off) { return static_cast<const char*>(q) + off; };
  // gate / up [n][I][K]: per expert, rows [p Is, (p+1) Is) are one
  // contiguous run of `per_row` bytes per row
  auto rows_slice = [&](const void* to, const void* from, size_t per_row) {
    for (size_t e = 0; e < n; ++e) {
      const size_t bytes = Is * per_row;
      if (cudaMemcpyAsync(static_cast<char*>(dst(to)) + e * bytes,
                          src(from, e * I * per_row + p * bytes), bytes,
                          cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return false;
    }
    return true;
  };
  // down [n][H][K = I]: every one of the n H rows keeps the bytes of columns
  // [p Is, (p+1) Is); `per_col` bytes per column (a fraction for codes)
  auto cols_slice = [&](const void* to, const void* from, size_t full_row, size_t slice_row) {
    return cudaMemcpy2DAsync(dst(to), slice_row, src(from, p * slice_row), full_row, slice_row,
                             n * H, cudaMemcpyDeviceToDevice, s) == cudaSuccess;
  };
  bool ok;
  if (!int4) {
    ok = rows_slice(slice->gate, full->gate, H * 2) && rows_slice(slice->up, full->up, H * 2) &&
         cols_slice(slice->down, full->down, I * 2, Is * 2);
  } else {
    ok = rows_slice(slice->gate, full->gate, H / 2) && rows_slice(slice->up, full->up, H / 2) &&
         rows_slice(slice->gate_scale, full->gate_scale, H / 32 * 2) &&
         rows_slice(slice->up_scale, full->up_scale, H / 32 * 2) &&
         cols_slice(slice->down, full->down, I / 2, Is / 2) &&
         cols_slice(slice->down_scale, full->down_scale, I / 32 * 2, Is / 32 * 2);
  }
  return ok ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_workspace_status(void* ws, moe_stream_t stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int code = 0;
  if (cudaMemcpyAsync(&code, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (code != 0 && cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  return code == 0 ? MOE_OK : (code == kStatusTimeout ? MOE_ERR_TIMEOUT : MOE_ERR_CUDA);
}

moe_status moe_debug_wait_timeout(void* ws, uint64_t budget_ns, moe_stream_t stream) {
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  moe_status st = check_device();
  if (st != MOE_OK) return st;
  return from_cuda(launch_wait_selftest(static_cast<int*>(ws), budget_ns,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Router + top-k without a caller workspace.
//
// For callers that cannot allocate device memory (an operator interface that
// passes only inputs and outputs, a loop that must not synchronise the device
// through cudaMalloc, a runtime whose pool gives nothing out), the router
// logits live in this fixed array instead of the workspace.  It is part of
// the library's device image, so every GPU that loads the library holds it
// (1 MiB) until the process exits.  All calls share it; overlapping calls
// race.  The logits are rewritten in full by every call before the top-k
// kernel reads them, so nothing in it needs clearing between calls.
static __device__ __align__(256) float g_static_router_logits[MOE_STATIC_ROUTER_LOGITS];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_scratch_mu;
struct StaticScratchAddr {
  unsigned long long ctx_id;  // unique id of the context the address belongs to
  float* addr;
};
StaticScratchAddr g_static_scratch_addr[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the current context (never reused within the process, so a
// device reset, which ends the context, also retires every address cached
// for it).
bool current_context_id(unsigned long long* id) {
  static const CtxGetCurrentFn get_current = []() -> CtxGetCurrentFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  static const CtxGetIdFn get_id = []() -> CtxGetIdFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<CtxGetIdFn>(p);
  }();
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_static_router_logits in the current device's context
// (host code only sees a host-side stand-in for the symbol).  Looked up with
// that device current the first time a context uses it, then cached under
// the context's id.
moe_status static_scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  // no context may be current yet on this thread: the lookup binds the
  // device's primary context, and the id is read after it
  unsigned long long ctx_id = 0;
  const bool have_id = current_context_id(&ctx_id);
  std::lock_guard<std::mutex> lock(g_static_scratch_mu);
  StaticScratchAddr& c = g_static_scratch_addr[dev];
  if (!have_id || !c.addr || c.ctx_id != ctx_id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_router_logits) != cudaSuccess || !p)
      return MOE_ERR_CUDA;
    if (!have_id && !current_context_id(&ctx_id)) return MOE_ERR_CUDA;
    c.addr = static_cast<float*>(p);
    c.ctx_id = ctx_id;
  }
  *out = c.addr;
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_router_topk_static_scratch(const moe_dims* d, const void* x,
                                                     const void* w_router, const float* b_router,
                                                     int32_t* topk_idx, float* topk_w,
                                                     moe_stream_t stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (d->T == 0) return MOE_OK;
  if (!x || !w_router || !b_router || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router)) return MOE_ERR_INVALID_ARG;
  if (static_cast<uint64_t>(d->T) * static_cast<uint64_t>(d->E) > MOE_STATIC_ROUTER_LOGITS)
    return MOE_ERR_WORKSPACE;
  if ((st = check_device()) != MOE_OK) return st;
  float* z = nullptr;
  if ((st = static_scratch_for_current_device(&z)) != MOE_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (launch_router_logits_simt(static_cast<const uint16_t*>(x),
                                static_cast<const uint16_t*>(w_router), b_router, z, d->T, d->H,
                                d->E, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return from_cuda(launch_topk(z, d->T, d->E, d->top_k, topk_idx, topk_w, s));
}
