// Grouped expert GEMMs over grouped-Int4 weights: in-kernel dequantisation
// into fp16 tensor-core operands (tcgen05 kind::f16, fp32 accumulation).
//
// Weights use the grouped fmt=4 Int4 format decoded as offset-binary,
// value = (nibble - 8) * scale ("feat(glm53): add device-resident HIP backend
// for MI350P", section "Key changes"), with one bf16 scale per 32 reduction
// elements.  (nibble - 8) * scale is exact in fp16 while the product stays
// in fp16's normal range (nibble - 8 has at most 3 significant bits and a
// bf16 scale 8, within fp16's 11), so the fp16 operand equals the decoded
// weight and the only rounding left is the fp32 accumulation.  Activations
// arrive as fp16 (x rows converted from bf16 by the permutation, exactly in
// fp16's normal range; h written as fp16 by gate/up).
//
// CTA = 15 warps, persistent over the same flat tile list as the bf16 path:
//   warp 0, lane 0   raw producer: TMA of packed codes (128-byte swizzle) and
//                    scales for 256 reduction elements per raw stage
//   warp 1           TMEM allocation; lane 0 issues tcgen05.mma
//   warps 2..5       epilogue (TMEM quadrant reads)
//   warps 6..13      dequantisers, two threads per weight row of the tile (one
//                    per matrix for gate/up, one per 32-element half for
//                    down); each turns code words into fp16 16-byte chunks
//                    written straight into the 128-byte-swizzled operand
//                    layout the MMA reads
//   warp 14, lane 0  activation producer: TMA of the token rows (fp16)
// Two A tiles per operand slot (NA = 2) are gate and up, or, for the down
// projection with the scatter-add epilogue, two 128-row blocks of the down
// weights against one token tile (256 output features per tile): each token
// tile then serves twice the weights and each commit twice the MMAs.
// The raw ring is as deep as shared memory allows (its stages are what carry
// the HBM bytes); two to four fp16 weight slots decouple dequantisation from
// the MMA; the activation tiles have a ring of their own, refilled as soon as
// the MMA has read them, so their loads run as far ahead as the code loads.
// Operand slots carry two barriers, one for the activation bytes (TMA) and
// one for the 128 dequantiser arrivals, so that after an abort every copy
// still in flight can be waited for on its own barrier.
#include <cuda_fp16.h>

#include "moe_kernels.h"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;                        // K per operand slot (one swizzle row of fp16)
constexpr int kRawK = 256;                     // K per raw stage
constexpr int kSubPerRaw = kRawK / kBK;        // 4
constexpr int kRowBytes = kBK * 2;             // 128
constexpr int kChunkRows = 16;
constexpr int kChunkBytes = kChunkRows * kRowBytes;
constexpr int kATileBytes = kBM * kRowBytes;   // 16 KB fp16 operand
constexpr int kCodeTileBytes = kBM * (kRawK / 2);  // 16 KB packed codes
constexpr int kScaleTileBytes = kBM * (kRawK / 32) * 2;  // 2 KB bf16 scales
constexpr int kBudget = 224 * 1024;
constexpr int kThreads = 480;
constexpr int kDqThread0 = 192;                // first dequantiser thread
constexpr int kDqThreads = 256;
constexpr int kDqWarpEnd = 14;                 // dequantiser warps are 6 .. 13
constexpr int kBWarp = 14;

__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }
constexpr int ceil_pow2_32(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <int BN, int NA>
struct Int4Cfg {
  static constexpr int kSlotBytes = NA * kATileBytes;
  static constexpr int kBTileBytes = BN * kRowBytes;
  static constexpr int kBStages = BN <= 16 ? 8 : (BN <= 64 ? 6 : 4);
  static constexpr int kBRingBytes = kBStages * kBTileBytes;
  static constexpr int kRawBytes = NA * (kCodeTileBytes + kScaleTileBytes);
  static constexpr int kRaw =
      cmin(NA == 2 ? 4 : 6, (kBudget - kBRingBytes - 2 * kSlotBytes) / kRawBytes);
  static constexpr int kSlots = cmin(4, (kBudget - kBRingBytes - kRaw * kRawBytes) / kSlotBytes);
  static constexpr int kAccStages = (2 * NA * BN <= 512) ? 2 : 1;
  static constexpr int kAccCols = NA * BN;
  static constexpr int kTmemCols = ceil_pow2_32(kAccStages * kAccCols);
  static constexpr int kSmemBytes = kSlots * kSlotBytes + kBRingBytes + kRaw * kRawBytes + 1024 + 512;
  static_assert(kSlotBytes % 1024 == 0 && kRawBytes % 1024 == 0 && kBTileBytes % 1024 == 0,
                "1024-byte alignment");
  static_assert(kSlots >= 2 && kRaw >= 2, "at least two operand slots and raw stages");
};

struct Int4Args {
  const int32_t* table;
  int K, N_out, mblocks, E, total_rows, out_rows;
  const int32_t* gather;
  const float* roww;
  float* out;      // down: scatter-add [T][N_out] or rows [rows][N_out]
  __half* h;       // gate/up: h [rows][N_out]
  int* status;
  uint64_t budget_ns;
};

// One 32-bit word of codes (element i of the word in bits 4i .. 4i+3) -> its
// eight fp16 weights (code - 8) * s as one 16-byte chunk, in the operand order
// of an aligned 8-element group: (e0, e4), (e1, e5), (e2, e6), (e3, e7).  In
// that order every pair is one mask-and-or (LOP3), no byte shuffles:
// (w & 0x000F000F) | 0x64006400 is the fp16 pair (1024 + e0, 1024 + e4), and
// (w & 0x00F000F0) | 0x54005400 is (64 + e1, 64 + e5), the nibble sitting four
// bits up where the ulp of 64 is 1/16.  Subtracting 1032 (or 72) leaves the
// integer e - 8 exactly; one multiply by the group scale rounds nothing
// while the product stays in fp16's normal range.
__device__ __forceinline__ uint4 dequant8(uint32_t w, __half2 s2) {
  const uint32_t w8 = w >> 8;
  const uint32_t p[4] = {(w & 0x000F000Fu) | 0x64006400u, (w & 0x00F000F0u) | 0x54005400u,
                         (w8 & 0x000F000Fu) | 0x64006400u, (w8 & 0x00F000F0u) | 0x54005400u};
  const __half2 off_lo = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  const __half2 off_hi = __halves2half2(__ushort_as_half(0x5480), __ushort_as_half(0x5480));
  uint32_t r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&p[i]), (i & 1) ? off_hi : off_lo);
    v = __hmul2(v, s2);
    r[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// 4 x 4 transpose across the four lanes 4j .. 4j+3 of a warp: lane 4j+r
// holds row r, (x0, x1, x2, x3) = M[r][0..3], and ends with column r,
// M[0..3][r].  Two exchange rounds (partner lane ^ 1, then ^ 2).
__device__ __forceinline__ void transpose4_lanes(float& x0, float& x1, float& x2, float& x3,
                                                 int lane) {
  const bool o1 = lane & 1, o2 = lane & 2;
  float s0 = __shfl_xor_sync(0xffffffffu, o1 ? x0 : x1, 1);
  float s1 = __shfl_xor_sync(0xffffffffu, o1 ? x2 : x3, 1);
  if (o1) {
    x0 = s0;
    x2 = s1;
  } else {
    x1 = s0;
    x3 = s1;
  }
  s0 = __shfl_xor_sync(0xffffffffu, o2 ? x0 : x2, 2);
  s1 = __shfl_xor_sync(0xffffffffu, o2 ? x1 : x3, 2);
  if (o2) {
    x0 = s0;
    x1 = s1;
  } else {
    x2 = s0;
    x3 = s1;
  }
}

__device__ __forceinline__ __half bf16_bits_to_half(uint32_t bits16) {
  return __float2half_rn(__uint_as_float(bits16 << 16));
}

template <int BN, int NA, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    int4_gemm_kernel(const __grid_constant__ CUtensorMap tm_c0,
                     const __grid_constant__ CUtensorMap tm_c1,
                     const __grid_constant__ CUtensorMap tm_s0,
                     const __grid_constant__ CUtensorMap tm_s1,
                     const __grid_constant__ CUtensorMap tm_sc0,
                     const __grid_constant__ CUtensorMap tm_sc1,
                     const __grid_constant__ CUtensorMap tm_ss0,
                     const __grid_constant__ CUtensorMap tm_ss1,
                     const __grid_constant__ CUtensorMap tm_b, const Int4Args a) {
  using Cfg = Int4Cfg<BN, NA>;
  // down with two row blocks per tile (rows 256 mb .. 256 mb + 255 of one matrix)
  constexpr bool kPair = NA == 2 && EPI == kEpiScatterAdd;
  constexpr int kTileRows = kPair ? 2 * kBM : kBM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* slots = base;
  uint8_t* bring = base + Cfg::kSlots * Cfg::kSlotBytes;
  uint8_t* raws = bring + Cfg::kBRingBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(raws + Cfg::kRaw * Cfg::kRawBytes);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + Cfg::kRaw;
  uint64_t* b_full = raw_empty + Cfg::kRaw;
  uint64_t* b_empty = b_full + Cfg::kBStages;
  uint64_t* a_full = b_empty + Cfg::kBStages;
  uint64_t* op_empty = a_full + Cfg::kSlots;
  uint64_t* tfull = op_empty + Cfg::kSlots;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::kRaw; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], kDqThreads);
    }
    for (int i = 0; i < Cfg::kBStages; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < Cfg::kSlots; ++i) {
      mbar_init(&a_full[i], kDqThreads);
      mbar_init(&op_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;
  const AbortState ab{abort_flag, a.status, a.budget_ns};

  pdl_wait();
  pdl_launch_dependents();
  const int total = a.table[0] * a.mblocks;
  const int KB = a.K / kBK;                       // operand slots per tile
  const int RB = (a.K + kRawK - 1) / kRawK;       // raw stages per tile

  auto code_tile = [&](int rs, int m) { return raws + rs * Cfg::kRawBytes + m * kCodeTileBytes; };
  auto scale_tile = [&](int rs, int m) {
    return raws + rs * Cfg::kRawBytes + NA * kCodeTileBytes + m * kScaleTileBytes;
  };
  auto a_tile = [&](int os, int m) { return slots + os * Cfg::kSlotBytes + m * kATileBytes; };
  auto b_tile = [&](int bs) { return bring + bs * Cfg::kBTileBytes; };

  if (warp == 0) {
    // ---------------------------------------------------------------- raw producer
    if (lane == 0) {
      // codes read by one token tile stream through L2 (evict_first); those
      // of a group cut into several token tiles (heavy experts, the shared
      // expert) are read again by its other tiles
      const uint64_t pol_once = policy_evict_first(), pol_again = policy_evict_last();
      int rs = 0;
      uint32_t rph = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileEntry te = table_entry(a.table, tile / a.mblocks);
        const int mb = tile % a.mblocks;
        const bool sh = te.group == a.E;
        const int ge = sh ? 0 : te.group;
        const uint64_t pol = te.ntiles > 1 ? pol_again : pol_once;
        for (int rb = 0; rb < RB; ++rb) {
          if (!mbar_wait(&raw_empty[rs], rph ^ 1u, ab)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&raw_full[rs], Cfg::kRawBytes);
          armed |= 1u << rs;
          armed_par = (armed_par & ~(1u << rs)) | (rph << rs);
          tma_load_3d(code_tile(rs, 0), sh ? &tm_sc0 : &tm_c0, &raw_full[rs], rb * (kRawK / 2),
                      mb * kTileRows, ge, pol);
          tma_load_3d(scale_tile(rs, 0), sh ? &tm_ss0 : &tm_s0, &raw_full[rs], rb * (kRawK / 32),
                      mb * kTileRows, ge, pol);
          if (NA == 2) {
            // gate/up: the up matrix; paired down: the second row block
            const int r1 = kPair ? mb * kTileRows + kBM : mb * kBM;
            tma_load_3d(code_tile(rs, 1), sh ? &tm_sc1 : &tm_c1, &raw_full[rs], rb * (kRawK / 2),
                        r1, ge, pol);
            tma_load_3d(scale_tile(rs, 1), sh ? &tm_ss1 : &tm_s1, &raw_full[rs],
                        rb * (kRawK / 32), r1, ge, pol);
          }
          if (++rs == Cfg::kRaw) {
            rs = 0;
            rph ^= 1u;
          }
        }
      }
      for (int s = 0; s < Cfg::kRaw; ++s)
        if ((armed >> s) & 1u) mbar_wait_drain(&raw_full[s], (armed_par >> s) & 1u);
    }
  } else if (warp == kBWarp) {
    // ---------------------------------------------------------------- activation producer
    if (lane == 0) {
      // activation rows: read by the mblocks tiles of their entry, which run
      // at about the same time; at prefill they exceed L2 (9 T K 2 bytes)
      const uint64_t pol = policy_evict_normal();
      int bs = 0;
      uint32_t bph = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileEntry te = table_entry(a.table, tile / a.mblocks);
        const int nchunks = (te.nrows + kChunkRows - 1) / kChunkRows;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&b_empty[bs], bph ^ 1u, ab)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&b_full[bs], nchunks * kChunkBytes);
          armed |= 1u << bs;
          armed_par = (armed_par & ~(1u << bs)) | (bph << bs);
          for (int c = 0; c < nchunks; ++c)
            tma_load_2d(b_tile(bs) + c * kChunkBytes, &tm_b, &b_full[bs], kb * kBK,
                        te.row0 + c * kChunkRows, pol);
          if (++bs == Cfg::kBStages) {
            bs = 0;
            bph ^= 1u;
          }
        }
      }
      for (int s = 0; s < Cfg::kBStages; ++s)
        if ((armed >> s) & 1u) mbar_wait_drain(&b_full[s], (armed_par >> s) & 1u);
    }
  } else if (warp >= 6 && warp < kDqWarpEnd) {
    // ---------------------------------------------------------------- dequantisers
    const int d = threadIdx.x - kDqThread0;
    const int r = d & (kBM - 1);             // weight row of the tile
    const int part = d >> 7;                 // gate/up: matrix; down: 32-element half
    const int sw = r & 7;                    // 128-byte swizzle phase of this row
    const int m = NA == 2 ? part : 0;
    constexpr int kHalves = NA == 2 ? 2 : 1; // 32-element groups per sub-block and thread
    // Byte offsets within the row of the swizzled 16-byte chunks this thread
    // reads (codes: chunk j = 32 elements = one scale group) and writes (fp16:
    // chunk c = 8 elements); the same for every stage and slot.
    uint32_t code_off[kSubPerRaw][kHalves], out_off[kHalves][4];
#pragma unroll
    for (int hh = 0; hh < kHalves; ++hh) {
      const int half = NA == 2 ? hh : part;
#pragma unroll
      for (int sb = 0; sb < kSubPerRaw; ++sb) code_off[sb][hh] = ((sb * 2 + half) ^ sw) << 4;
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) out_off[hh][wd] = ((half * 4 + wd) ^ sw) << 4;
    }
    int rs = 0, os = 0;
    uint32_t rph = 0, oph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      for (int rb = 0; ok && rb < RB; ++rb) {
        if (!mbar_wait(&raw_full[rs], rph, ab)) {
          ok = false;
          break;
        }
        // eight bf16 scales of this row's 256 elements: group j in word j / 2
        const uint4 sv = *reinterpret_cast<const uint4*>(scale_tile(rs, m) + r * 16);
        const uint32_t sw4[4] = {sv.x, sv.y, sv.z, sv.w};
        const uint8_t* ct = code_tile(rs, m) + r * 128;
        // K is a multiple of the raw stage (256), so every stage holds kSubPerRaw slots
#pragma unroll
        for (int sb = 0; sb < kSubPerRaw; ++sb) {
          if (!mbar_wait(&op_empty[os], oph ^ 1u, ab)) {
            ok = false;
            break;
          }
          uint8_t* at = a_tile(os, m) + r * kRowBytes;
#pragma unroll
          for (int hh = 0; hh < kHalves; ++hh) {
            const int shift = (NA == 2 ? hh : part) * 16;  // group 2 sb + half
            const __half s1 = bf16_bits_to_half((sw4[sb] >> shift) & 0xFFFFu);
            const __half2 s2 = __halves2half2(s1, s1);
            const uint4 cw = *reinterpret_cast<const uint4*>(ct + code_off[sb][hh]);
            *reinterpret_cast<uint4*>(at + out_off[hh][0]) = dequant8(cw.x, s2);
            *reinterpret_cast<uint4*>(at + out_off[hh][1]) = dequant8(cw.y, s2);
            *reinterpret_cast<uint4*>(at + out_off[hh][2]) = dequant8(cw.z, s2);
            *reinterpret_cast<uint4*>(at + out_off[hh][3]) = dequant8(cw.w, s2);
          }
          fence_proxy_async_smem();
          mbar_arrive(&a_full[os]);
          if (++os == Cfg::kSlots) {
            os = 0;
            oph ^= 1u;
          }
        }
        mbar_arrive(&raw_empty[rs]);
        if (++rs == Cfg::kRaw) {
          rs = 0;
          rph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc0 = idesc_f16(kBM, 16, false) & ~(0x3Fu << 17);
      int os = 0, bs = 0, acc = 0;
      uint32_t oph = 0, bph = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileEntry te = table_entry(a.table, tile / a.mblocks);
        const uint32_t idesc = idesc0 | (static_cast<uint32_t>(round16(te.nrows) >> 3) << 17);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, ab)) break;
        tc_fence_after_sync();
        const uint32_t d0 = tmem_base + acc * Cfg::kAccCols;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&b_full[bs], bph, ab) || !mbar_wait(&a_full[os], oph, ab)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t db = sw128_kmajor_desc(smem_u32(b_tile(bs)));
          const uint64_t da0 = sw128_kmajor_desc(smem_u32(a_tile(os, 0)));
          const uint64_t da1 = sw128_kmajor_desc(smem_u32(a_tile(os, NA - 1)));
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint32_t accum = (kb | k) != 0;
            umma_f16(d0, da0 + 2 * k, db + 2 * k, idesc, accum);
            if (NA == 2) umma_f16(d0 + BN, da1 + 2 * k, db + 2 * k, idesc, accum);
          }
          umma_commit(&op_empty[os]);
          umma_commit(&b_empty[bs]);
          if (++os == Cfg::kSlots) {
            os = 0;
            oph ^= 1u;
          }
          if (++bs == Cfg::kBStages) {
            bs = 0;
            bph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        if (Cfg::kAccStages == 2) {
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        } else {
          acc_phase ^= 1u;
        }
      }
      umma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    // the scatter-add's output lines receive one addition per (token, slot)
    // spread over the launch: kept resident in L2 between them
    const uint64_t pol_out = policy_evict_last();
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const TileEntry te = table_entry(a.table, tile / a.mblocks);
      const int mb = tile % a.mblocks;
      // Scatter-add: the tile's token ids and routing weights (nrows <= BN
      // <= 128), loaded while its MMAs run -- lane l holds rows l, l + 32,
      // l + 64, l + 96 -- so the atomics below wait on no global load.
      int tk[4] = {-1, -1, -1, -1};
      float tw[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (EPI == kEpiScatterAdd) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = j * 32 + lane;
          const int rr = te.row0 + i;
          if (i < te.nrows && rr < a.total_rows) {
            const int t = a.gather[rr];
            tw[j] = a.roww[rr];
            tk[j] = (t >= 0 && t < a.out_rows) ? t : -1;
          }
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, ab))) break;
      tc_fence_after_sync();
      const int f = mb * kTileRows + q * 32 + lane;
      // column of feature f in the down GEMM's operand order (see dequant8)
      const int f_op = (f & ~7) | ((f & 3) << 1) | ((f >> 2) & 1);
      const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * Cfg::kAccCols;
      const int n = round16(te.nrows);
      for (int c0 = 0; c0 < n; c0 += 16) {
        uint32_t v0[16], v1[16];
        tmem_ld_32x32b_x16(tq + c0, v0);
        if (NA == 2) tmem_ld_32x32b_x16(tq + BN + c0, v1);
        tmem_ld_wait();
        if (EPI == kEpiScatterAdd) {
          // Lanes 4j .. 4j+3 hold four consecutive features; a 4 x 4 exchange
          // leaves lane 4j+r with those four features of token column
          // 4g + r, added with one 16-byte atomic instead of four scalar ones.
          // Paired down: the second block's features are 128 further on.
          const int r4 = lane & 3;
#pragma unroll
          for (int blk = 0; blk < (kPair ? 2 : 1); ++blk) {
            const int fb = f + blk * kBM;
            float* const ob = a.out + (fb & ~3);
            const uint32_t* v = blk ? v1 : v0;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              float x0 = __uint_as_float(v[4 * g]), x1 = __uint_as_float(v[4 * g + 1]);
              float x2 = __uint_as_float(v[4 * g + 2]), x3 = __uint_as_float(v[4 * g + 3]);
              transpose4_lanes(x0, x1, x2, x3, lane);
              const int cb = c0 + 4 * g;  // a multiple of 4: the same register slot for all lanes
              const int j = cb >> 5;
              const int src = (cb + r4) & 31;
              const int t = __shfl_sync(
                  0xffffffffu, j == 0 ? tk[0] : j == 1 ? tk[1] : j == 2 ? tk[2] : tk[3], src);
              const float wr = __shfl_sync(
                  0xffffffffu, j == 0 ? tw[0] : j == 1 ? tw[1] : j == 2 ? tw[2] : tw[3], src);
              const int c = cb + r4;
              if (c < te.nrows && fb < a.N_out) {
                if (t >= 0)
                  red_add_f32x4(ob + static_cast<size_t>(t) * a.N_out,
                                make_float4(wr * x0, wr * x1, wr * x2, wr * x3), pol_out);
              }
            }
          }
        } else if (f < a.N_out) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = c0 + i;
            const int rr = te.row0 + c;
            if (c < te.nrows && rr < a.total_rows) {
              const float d = __uint_as_float(v0[i]);
              if (NA == 2) {
                const float hv = clamped_swiglu(d, __uint_as_float(v1[i]));
                a.h[static_cast<size_t>(rr) * a.N_out + f_op] = __float2half_rn(hv);
              } else {
                a.out[static_cast<size_t>(rr) * a.N_out + f] = d;
              }
            }
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&tempty[acc]);
      if (Cfg::kAccStages == 2) {
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      } else {
        acc_phase ^= 1u;
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

template <int BN, int NA, int EPI>
cudaError_t int4_dispatch(const Int4Launch& L, cudaStream_t s) {
  using Cfg = Int4Cfg<BN, NA>;
  auto kern = int4_gemm_kernel<BN, NA, EPI>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (err != cudaSuccess) return err;
  Int4Args a{L.table, L.K, L.N_out, L.mblocks, L.E, L.total_rows, L.out_rows,
             L.gather, L.roww, L.out, static_cast<__half*>(L.h), L.status, L.budget_ns};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, L.tm_c[0], L.tm_c[1], L.tm_s[0], L.tm_s[1], L.tm_sc[0],
                            L.tm_sc[1], L.tm_ss[0], L.tm_ss[1], L.tm_b, a);
}

template <int NA, int EPI>
cudaError_t int4_by_bn(const Int4Launch& L, cudaStream_t s) {
  switch (L.BN) {
    case 16: return int4_dispatch<16, NA, EPI>(L, s);
    case 32: return int4_dispatch<32, NA, EPI>(L, s);
    case 64: return int4_dispatch<64, NA, EPI>(L, s);
    case 128: return int4_dispatch<128, NA, EPI>(L, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_int4_gemm(const Int4Launch& L, cudaStream_t s) {
  if (L.na == 2)
    return L.epilogue == kEpiScatterAdd ? int4_by_bn<2, kEpiScatterAdd>(L, s)
                                        : int4_by_bn<2, kEpiStoreRows>(L, s);
  if (L.epilogue == kEpiScatterAdd) return int4_by_bn<1, kEpiScatterAdd>(L, s);
  return int4_by_bn<1, kEpiStoreRows>(L, s);
}

}  // namespace moe
