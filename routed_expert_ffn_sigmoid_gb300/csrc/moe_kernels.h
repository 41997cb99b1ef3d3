// Internal launch interface between the C-ABI translation unit and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

constexpr int kMaxE = 512;        // routed experts supported by router / permute
constexpr int kMaxTopK = 16;
constexpr int kPermTokBlock = 128; // tokens per counting-sort block
constexpr int kTableHeaderBytes = 16;
constexpr int kSmallT = 128;       // tokens handled by the one-CTA routing kernel
constexpr int kSmallThreads = 512;

// One grouped-GEMM work entry: rows [row0, row0 + nrows) of group `group`
// (group == E is the shared expert).  nrows <= the launch's token tile BN.
// ntiles: the number of entries of the group, so that a kernel knows
// whether other tiles will read the same weights (L2 policy).
struct TileEntry {
  int32_t group, row0, nrows, ntiles;
};

// ---------------------------------------------------------------- router

// z[t][e] = sum_h x[t][h] w_router[e][h] + b[e] on CUDA cores (fp32 FMA).
cudaError_t launch_router_logits_simt(const uint16_t* x, const uint16_t* w_router, const float* b,
                                      float* z, int T, int H, int E, cudaStream_t s);

// Per token: top_k of z (ties to the lower index), sigmoid, renormalise.
// The router kernels also clear zero_n floats of zero_out (the layer output,
// when the down epilogue adds into it) with their whole grid.
// Decode-size router: partial logits per reduction slice of kRouterSliceK
// elements, part [slices][T][E] fp32, then per token the slice sum in slice
// order + bias and the top-k (z [T][E] also written when z != nullptr).
constexpr int kRouterSliceK = 256;
inline int router_slices(int H) { return (H + kRouterSliceK - 1) / kRouterSliceK; }
cudaError_t launch_router_partials(const uint16_t* x, const uint16_t* w_router, float* part,
                                  int T, int H, int E, float* zero_out, size_t zero_n,
                                  cudaStream_t s);
// Outputs of the decode-size permutation (T <= kSmallT), which the last CTA
// of the top-k kernel runs once every token's selection is written; `done`
// is a counter that is zero before the launch and zero again after it.
struct SmallPermOut {
  int* done;
  int BN;
  int32_t* offsets;
  int32_t* gather;
  int32_t* row_of;
  float* roww;
  int32_t* table;
  int32_t* table2;  // optional second tile table with entries of at most BN2 rows
  int BN2;
};
cudaError_t launch_router_reduce_topk(const float* part, const float* b, int T, int H, int E,
                                      int k, int32_t* idx, float* w, float* z,
                                      const SmallPermOut* perm, cudaStream_t s);
// Routing of up to kRouteSmallT tokens (H <= 4096) in one launch: logits
// (z [T][E], workspace), top-k (idx / w) and, in the last CTA to finish, the
// permutation into `perm` (done: a counter that is zero before the launch
// and zero again after it).  Also clears zero_n floats of zero_out.
constexpr int kRouteSmallT = 16;
cudaError_t launch_route_small(const uint16_t* x, const uint16_t* w_router, const float* b, int T,
                               int H, int E, int k, float* z, int32_t* idx, float* w,
                               const SmallPermOut& perm, float* zero_out, size_t zero_n,
                               cudaStream_t s);
// The same permutation as a one-CTA launch of its own (`done` unused).
cudaError_t launch_small_permutation(const int32_t* idx, const float* w, int T, int E, int k,
                                     const SmallPermOut& p, cudaStream_t s);
cudaError_t launch_topk(const float* z, int T, int E, int k, int32_t* idx, float* w,
                        cudaStream_t s, float* zero_out = nullptr, size_t zero_n = 0);

// ---------------------------------------------------------------- permute

cudaError_t launch_perm_count(const int32_t* idx, int T, int E, int k, int32_t* blockcnt,
                              cudaStream_t s);
// Turns block counts into per-block row bases, writes offsets[E+2] and the
// tile table (entries of at most BN rows).  One CTA.
cudaError_t launch_perm_scan(int32_t* blockcnt, int T, int E, int k, int32_t* offsets,
                             int32_t* table, int BN, cudaStream_t s);
// Stable ranks inside each block; gather / row_of / row weights.
cudaError_t launch_perm_scatter(const int32_t* idx, const float* w, const int32_t* blockbase,
                                int T, int E, int k, int32_t* gather, int32_t* row_of,
                                float* roww, cudaStream_t s);
// x_perm[row_of[t][j]] = x[t] for j < k and x_perm[k*T + t] = x[t] (the
// shared row; k = 0: x_perm = x), in token order; to_fp16 converts bf16 ->
// fp16 in the Int4 operand order on the way.  When zero_out is not null the
// kernel also zeroes zero_n floats there (a multiple of 4, 16-byte aligned).
cudaError_t launch_scatter_rows(const uint16_t* x, const int32_t* row_of, int T, int H, int k,
                                bool to_fp16, uint16_t* x_perm, float* zero_out, size_t zero_n,
                                cudaStream_t s);
// The same copy of each token's row into its k + 1 permuted rows, as two
// e4m3 planes under a power-of-two scale sigma per token (max |x sigma| in
// [128, 256)): x8[2r][.] = e4m3(x sigma), x8[2r + 1][.] = e4m3(x sigma -
// hi), each aligned group of 8 columns in the order (0, 1, 4, 5, 2, 3, 6, 7),
// xinv[r] = 1 / sigma.  Also clears zero_n floats of zero_out.
cudaError_t launch_split_rows_e4m3(const uint16_t* x, const int32_t* row_of, int T, int H, int k,
                                   uint8_t* x8, float* xinv, float* zero_out, size_t zero_n,
                                   cudaStream_t s);
// Dense FFN: rows 0..T-1 are one group (group 0): gather[r] = r, roww[r] = 1
// and a tile table of ceil(T / BN) entries.
cudaError_t launch_dense_rows(int T, int BN, int32_t* gather, float* roww, int32_t* table,
                              cudaStream_t s);
// Tile table from existing offsets (for the unfused expert entry point);
// at most `capacity` entries.
cudaError_t launch_table_from_offsets(const int32_t* offsets, int E, int rows, int capacity,
                                      int32_t* table, int BN, cudaStream_t s);

// ---------------------------------------------------------------- combine

cudaError_t launch_combine(const float* y_perm, const int32_t* row_of, const float* w, int T,
                           int H, int k, bool accumulate, float* out, cudaStream_t s);

// ---------------------------------------------------------------- grouped GEMMs

struct GateUpLaunch {
  CUtensorMap tm_gate, tm_up, tm_sgate, tm_sup, tm_x;
  // shared expert first (fused layer): n_sh > 0 entries of the shared group
  // (rows sh_row0 + t, tokens x[t] through tm_xs: x [T][K], 16-row boxes)
  // run before the kernel waits for the routing
  CUtensorMap tm_xs;
  int n_sh, T, sh_row0;
  const int32_t* table;
  const int32_t* xrows;  // null: tm_x maps x_perm (16-row boxes); else tm_x maps x
                         // (1-row boxes) and row r of the tile is x[xrows[r]]
  int BN;            // token tile (16, 32, 64, 128, 256)
  int K;             // H
  int I;             // intermediate size (features)
  int E;             // group id of the shared expert
  int a_rows;        // rows of one weight box (min(128, I))
  int total_rows;    // rows of x_perm / h (stores beyond are dropped)
  int ksplit;        // K-split units per tile (1 = none); > 1 needs partial + counters
  float* partial;    // [units][2][BN][128] fp32 partial G/U
  int* counters;     // [tiles] finished-unit counters, zero between calls
  bool bf16;         // bf16 operands (else fp16)
  void* h0;          // bf16 path: hi plane; fp16 path: h
  void* h1;          // bf16 path: lo plane; fp16 path: null
  int* status;
  uint64_t budget_ns;
  int grid;
};
cudaError_t launch_gateup(const GateUpLaunch& L, cudaStream_t s);

enum DownEpilogue : int { kEpiScatterAdd = 0, kEpiStoreRows = 1, kEpiRouter = 2 };

// The decode FFN of a fused layer call in one persistent launch (bf16
// weights, weights-as-M tiles of BN <= 64 token rows, scatter-add output):
// every gate/up unit, then every down unit, with per-entry counters in
// place of the kernel boundary.  g describes the gate/up half (n_sh > 0:
// the shared expert's entries come first); the down half reads h through
// tm_h0 / tm_h1 (16-row boxes) and the down weights through tm_down /
// tm_sdown.  ready: n_ready + 2 ints (per-entry counters, finished CTAs,
// the unit queue's counter), zero before the launch and zero again after it.  grid must not exceed the SM count (the units wait on one
// another across CTAs).
struct FfnLaunch {
  struct GateUpLaunch g;
  CUtensorMap tm_down, tm_sdown, tm_h0, tm_h1;
  int ks_d;          // K-split units per down tile (1 = none)
  int* ready;
  int n_ready;
  const int32_t* gather;
  const float* roww;
  float* out;        // [T][H], added into
  int out_rows;
  int grid;
};
cudaError_t launch_decode_ffn(const FfnLaunch& L, cudaStream_t s);

struct DownLaunch {
  CUtensorMap tm_a, tm_a_shared, tm_b0, tm_b1;
  const int32_t* table;  // null: dense tiles over `dense_rows` rows, group 0
  int dense_rows;
  int BN;
  int nb;            // B operands per k-step: 2 = split (hi + lo), 1 = single
  int K;             // reduction length
  int N_out;         // output features (H for down, E for the router)
  int mblocks;       // ceil(N_out / 128)
  int E;             // shared group id (-1 when there is none)
  int a_rows;        // rows of one weight box
  int total_rows;    // rows of the B operand (stores beyond are dropped)
  int out_rows;      // scatter-add: tokens in out (gather ids beyond are dropped)
  int ksplit;        // K-split units per tile, scatter-add epilogue only (1 = none)
  bool bf16;
  int epilogue;      // DownEpilogue
  const int32_t* gather;
  const float* roww;
  const float* bias;
  float* out;        // scatter-add: [T][N_out]; store rows: [rows][N_out]
  int* status;
  uint64_t budget_ns;
  int grid;
};
cudaError_t launch_down(const DownLaunch& L, cudaStream_t s);

// Grouped GEMM over grouped-Int4 weights (dequantised in-kernel to fp16).
// na = 2, store rows: gate/up with the clamped SwiGLU, h written as fp16
// [rows][N_out]; na = 2, scatter-add: down over tiles of two 128-row blocks
// (mblocks = N_out / 256; tm_c[1] = tm_c[0], the same for the scales);
// na = 1: down with the scatter-add or store-rows epilogue.
struct Int4Launch {
  CUtensorMap tm_c[2], tm_s[2];    // codes / scales of the routed stacks
  CUtensorMap tm_sc[2], tm_ss[2];  // codes / scales of the shared expert
  CUtensorMap tm_b;                // fp16 activation rows
  const int32_t* table;
  int BN, na, K, N_out, mblocks, E, total_rows, out_rows, epilogue;
  const int32_t* gather;
  const float* roww;
  float* out;
  void* h;
  int* status;
  uint64_t budget_ns;
  int grid;
};
cudaError_t launch_int4_gemm(const Int4Launch& L, cudaStream_t s);

// Int4 grouped GEMMs on 8-bit operands (decode sizes): codes n - 8 as e5m2
// against the activation rows as e4m3 planes under power-of-two scales, each
// aligned group of 8 elements in the order (0, 1, 4, 5, 2, 3, 6, 7) on both
// sides; one MMA per scale group, scales applied by the epilogue.
//   na = 2: gate/up with the clamped SwiGLU.  B: x as two planes (hi, lo),
//           binv [rows] = 1 / sigma; tile entries of at most kF8MaxRows rows.
//           Writes h as three planes h8 [rows][3][N_out] (hi, mid, lo) and
//           hinv [rows][N_out / 32] = 1 / sigma per group of 32 features.
//   na = 1: down with the scatter-add or store-rows epilogue.  B: those h
//           planes, binv = hinv; tile entries of at most kF8DownMaxRows rows.
//   na = 2 with the scatter-add epilogue: the same down over tiles of two
//           128-row blocks (N_out % 256 == 0; tm_c[1] = tm_c[0], scale[1] =
//           scale[0], the same for the shared expert).
constexpr int kF8MaxRows = 8;
constexpr int kF8DownMaxRows = 5;
struct Int4F8Launch {
  CUtensorMap tm_c[2];   // codes of the routed stacks (gate, up; or down)
  CUtensorMap tm_sc[2];  // codes of the shared expert
  CUtensorMap tm_b;      // e4m3 activation planes, row P r + p
  const int32_t* table;
  int na, epilogue, K, N_out, E, total_rows, out_rows;
  const void* scale[2];   // bf16 [E][N_out][K / 32]
  const void* sscale[2];  // bf16 [1][N_out][K / 32]
  const float* binv;
  uint8_t* h8;
  float* hinv;
  const int32_t* gather;
  const float* roww;
  float* out;
  int* status;
  uint64_t budget_ns;
  int grid;
};
cudaError_t launch_int4_f8_gemm(const Int4F8Launch& L, cudaStream_t s);

// Int4 grouped GEMVs on CUDA cores (decode sizes): 8-bit integer dot products
// of the codes against the activation rows quantised to 16 bits (a signed
// high and an unsigned low byte) under a power-of-two scale per row and group
// of 32; tile entries of at most kGemvMaxRows rows.  Shapes: K = H a multiple
// of 1024 up to 4096, I a multiple of 512 up to 2048 (int4_gemv_shape_ok).
//   gate/up: token rows x[xrows[r]] (bf16 [.][K]), N_out = I; writes h as
//            planes hq [rows][4][I / 32] x 16 bytes, the scales hs [rows][I / 32]
//            and 8 sum q hc [rows][I / 32].
//   down:    K = I, N_out = H; reads those planes; scatter-add (out [out_rows][H]
//            += roww[r] y, token gather[r]) or store rows (out = y_perm [rows][H]).
// codes[1] / scale[1] / scodes[1] / sscale[1] are unused by down.
constexpr int kGemvMaxRows = 8;
struct Int4GemvLaunch {
  const int32_t* table;
  int epilogue, K, N_out, E, total_rows, out_rows, grid;
  const uint16_t* x;
  const int32_t* xrows;
  const void* codes[2];    // routed stacks [E][N_out][K / 2]
  const void* scale[2];    // bf16 [E][N_out][K / 32]
  const void* scodes[2];   // the shared expert's
  const void* sscale[2];
  uint8_t* hq;
  float* hs;
  int32_t* hc;
  const int32_t* gather;
  const float* roww;
  float* out;
};
bool int4_gemv_shape_ok(int H, int I);
cudaError_t launch_int4_gemv_gateup(const Int4GemvLaunch& L, cudaStream_t s);
cudaError_t launch_int4_gemv_down(const Int4GemvLaunch& L, cudaStream_t s);

// Token-major grouped GEMM (bf16, token tiles of 128 rows): gate/up with the
// SwiGLU epilogue (h hi/lo planes) or down with the scatter-add / store-rows
// epilogue.  tm_a: token planes (x_perm; or h hi, h lo), tm_b / tm_sb: weight
// stacks of the routed / shared experts (gate, up; or down).
struct TmLaunch {
  CUtensorMap tm_a[2], tm_b[2], tm_sb[2];
  const int32_t* table;
  const int32_t* arows;  // gate/up: non-null -> token row r is x[arows[r]], copied from
  const void* xsrc;      // xsrc [T][xpitch] bf16 by the producer warp (tm_a[0] unused)
  int xpitch;
  float* zero_out;       // gate/up: zero_n floats the kernel clears (null: none)
  size_t zero_n;
  bool gateup;
  int K, N_out, nblocks, E, total_rows, out_rows, epilogue;
  const int32_t* gather;
  const float* roww;
  float* out;
  void* h0;
  void* h1;
  int* status;
  uint64_t budget_ns;
  int grid;
};
cudaError_t launch_tm_gemm(const TmLaunch& L, cudaStream_t s);

// Diagnostic bounded wait on a barrier nothing completes.
cudaError_t launch_wait_selftest(int* status, uint64_t budget_ns, cudaStream_t s);

}  // namespace moe
