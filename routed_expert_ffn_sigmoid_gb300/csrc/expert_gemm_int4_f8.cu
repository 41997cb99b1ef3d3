// Grouped expert GEMMs over grouped-Int4 weights on 8-bit tensor-core
// operands, for decode-size groups: gate/up with the clamped SwiGLU (NA = 2)
// and down with the routing weight and the scatter-add (NA = 1).
//
// Weights use the grouped fmt=4 Int4 format decoded as offset-binary,
// value = (nibble - 8) * scale ("feat(glm53): add device-resident HIP backend
// for MI350P", section "Key changes"), one bf16 scale per 32 reduction
// elements; the expert FFN follows "Add GLM-5.3-Flash (glm5next) support
// with ROCmFP mix qtypes (105/106)", section "MoE FFN (REAL routed expert
// execution)".
//
// Why 8-bit operands.  With fp16 operand tiles the Int4 GEMM is bound by
// shared memory: per weight the dequantisers store 2 bytes and the tensor
// core reads 2 more.  Here the code n - 8 (an integer in [-8, 7], exact in
// e5m2) is the A operand, 1 byte per weight, and the scale is applied after
// the product:
//   sum_k (n_k - 8) s_g b_k = s_g * sum_{k in g} (n_k - 8) b_k,
// so each MMA covers exactly one scale group (K = 32 for kind::f8f6f4) into an
// accumulator of its own, and the epilogue warps add s_g times it into
// registers.  The activation rows (B) enter as e4m3 planes under a power-of-
// two scale, each plane the rounding remainder of the ones before:
//   gate/up: x as hi + lo, one scale per token row: bf16's 8 significant
//            bits split exactly into 4 + 4 for values at least 2^-9 of the
//            row's largest |x|; below that lo reaches e4m3's subnormal
//            quantum and the error stays under 2^-17 of the largest |x|;
//   down:    h as hi + mid + lo, one scale per token row and group of 32
//            features, chosen by the gate/up epilogue from the largest |h| of
//            the group: 12 significant bits for values within 2^-5 of that
//            largest |h|, an absolute error below 2^-17 of it for the rest
//            (where the last plane reaches e4m3's subnormal quantum).
// Every product is exact in fp32; only fp32 accumulation rounds.
//
// B operand: rows P t .. P t + P - 1 are token t's planes (P = 2 or 3), so
// N = 16 covers 8 (gate/up) or 5 (down) tokens; columns past the tile
// entry's rows are ignored.  Along K both operands hold each aligned group of
// 8 elements in the order (0, 1, 4, 5, 2, 3, 6, 7), the order the weight
// bytes come out of e5m2_of_codes8.
//
// CTA = 16 warps, persistent over the flat tile list:
//   warp 0, lane 0   code producer: TMA of the packed codes, 256 reduction
//                    elements per raw stage
//   warps 1, 15      lane 0 of each issues tcgen05.mma kind::f8f6f4 (A e5m2
//                    from TMEM, B e4m3 from shared memory): one matrix each
//                    (gate/up) or two of a slot's scale groups each (down);
//                    warp 1 also allocates TMEM
//   warps 2..5       epilogue: per operand slot (four scale groups),
//                    tcgen05.ld of the accumulator columns that hold tokens,
//                    scale and add; after the last group the SwiGLU and the
//                    h planes (gate/up) or the scatter-add / row store (down)
//   warps 6..13      dequantisers, two threads per weight row (one per matrix
//                    for gate/up, one per two of a slot's four groups for
//                    down; a warp's rows are its TMEM lane quadrant): code
//                    words -> e5m2 bytes (fp16 mask-and-or, one half2
//                    subtract, one byte permute per four codes), stored into
//                    the operand slot's TMEM columns (tcgen05.st)
//   warp 14, lane 0  activation producer: TMA of the e4m3 planes, four
//                    operand slots' B tiles per stage
// TMEM holds the operand slots and a ring of accumulator entries, one entry
// (four scale groups) per slot.  Per slot the issuers commit once each to the
// entry's barrier; the epilogue waits on it, and so do the dequantisers
// before they overwrite the slot's operand columns two slots later (the same
// MMAs read them), which spares a commit per slot.  Why the operand is in
// TMEM and the issue is split: measured on GB300, a 128 x 16 x 32 MMA costs
// ~44 cycles to issue, tcgen05.st moves ~250 B per cycle per SM next to MMAs
// without slowing them, and a commit costs ~200 cycles in this kernel; with
// the operand in shared memory the kernel moved ~3 B of shared memory per
// weight.  Every wait is bounded as in the other GEMM kernels.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <type_traits>

#include "moe_kernels.h"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;
constexpr int kSlotK = 128;                        // 8-bit elements per 128-byte swizzle row
constexpr int kRawK = 256;                         // reduction elements per raw stage
constexpr int kSlotsPerRaw = kRawK / kSlotK;       // 2
constexpr int kGroupsPerSlot = kSlotK / 32;        // 4
constexpr int kCodeTileBytes = kBM * (kRawK / 2);  // 16 KB packed codes per matrix
constexpr int kBRows = 16;
constexpr int kBTileBytes = kBRows * kSlotK;       // 2 KB: one operand slot's B tile
constexpr int kBSub = 4;                           // slots (B tiles) per B stage
constexpr int kBStageBytes = kBSub * kBTileBytes;  // 8 KB
constexpr int kBStages = 4;
constexpr int kGroupsPerSync = 4;                  // groups per accumulator handshake (a slot)
constexpr int kGroupsPerLoad = 2;                  // groups per TMEM load batch of the epilogue
constexpr int kTmemCols = 512;
constexpr int kBarBytes = 1024;
constexpr int kThreads = 512;
constexpr int kDqThread0 = 192;
constexpr int kDqThreads = 256;
constexpr int kDqWarpEnd = 14;
constexpr int kBWarp = 14;
// The MMAs are issued by two threads on different SM sub-partitions (warps 1
// and 15), each for one matrix (gate/up) or two of a slot's four scale
// groups (down): a single issuer shares its sub-partition with two
// dequantiser warps and loses issue slots to their ALU work (measured: 8
// MMAs plus bookkeeping took ~1.6k cycles per slot, against ~0.4k alone).
constexpr int kMmaWarp1 = 15;
constexpr int kIssuers = 2;
constexpr int kMaxGroups = 128;                    // K / 32 of the down projection (I <= 4096)

// NA: weight matrices (A tiles) per operand slot -- gate and up, or for the
// down projection two 128-row blocks of the down weights against one h tile
// (kDown with NA = 2) -- or one (down).
template <int NA, bool kDown>
struct F8Cfg {
  static constexpr int kPlanes = kDown ? 3 : 2;               // B rows per token
  static constexpr int kMaxTok = kBRows / kPlanes;            // 5 or 8
  static constexpr int kGroupCols = 16 * NA;                  // accumulator columns per group
  static constexpr int kEntryCols = kGroupsPerSync * kGroupCols;
  // TMEM: the accumulator ring first, then the operand slots (A, e5m2:
  // 128 lanes x 32 bytes = 8 columns per scale group and matrix)
  static constexpr int kSlots = NA == 2 ? 2 : 3;
  static constexpr int kACols = NA * kGroupsPerSlot * 8;      // 64 or 32
  static constexpr int kAccRing = (kTmemCols - kSlots * kACols) / kEntryCols;  // 3 or 6
  static constexpr int kABase = kAccRing * kEntryCols;
  static constexpr int kRawBytes = NA * kCodeTileBytes;
  static constexpr int kRaw = NA == 2 ? 5 : 10;
  static constexpr int kSmemBytes = kRaw * kRawBytes + kBStages * kBStageBytes + 1024 + kBarBytes;
  static_assert(kSmemBytes <= 227 * 1024 - (kDown ? 4 * kF8DownMaxRows * kMaxGroups * 4 : 0),
                "shared memory");
  static_assert(kABase + kSlots * kACols <= kTmemCols, "TMEM columns");
  static_assert(kMaxTok == (kDown ? kF8DownMaxRows : kF8MaxRows), "tile entry rows");
  // one accumulator entry per operand slot: the dequantisers reuse slot n's
  // TMEM columns once acc_full of the entry of slot n - kSlots has completed
  static_assert(kGroupsPerSync == kGroupsPerSlot, "one accumulator entry per slot");
  static_assert(kSlots < kAccRing, "an entry is reused only after its slot's reuse");
};

struct F8Args {
  const int32_t* table;
  int K, N_out, mblocks, E, total_rows, out_rows;
  const uint16_t* scale0;   // routed scales [E][N_out][K / 32] bf16 (gate, or down)
  const uint16_t* scale1;   // (up)
  const uint16_t* sscale0;  // shared expert [1][N_out][K / 32]
  const uint16_t* sscale1;
  const float* binv;        // gate/up: [rows] 1 / sigma; down: [rows][K / 32]
  uint8_t* h8;              // gate/up: h planes [rows][3][N_out]
  float* hinv;              // gate/up: [rows][N_out / 32]
  const int32_t* gather;    // down
  const float* roww;
  float* out;               // down: scatter-add [T][N_out] or rows [rows][N_out]
  int* status;
  uint64_t budget_ns;
};

// Byte permute: bytes 0..3 of a, 4..7 of b, four 4-bit selectors in c[15:0].
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// One 32-bit word of codes (code i in bits 4i .. 4i+3) -> eight e5m2 bytes
// of code - 8, in the operand order (0, 1, 4, 5, 2, 3, 6, 7) of the group
// of 8.  (w & 0x000F000F) | 0x64006400 is the fp16 pair (1024 + c0,
// 1024 + c4) and (w & 0x00F000F0) | 0x54005400 is (64 + c1, 64 + c5);
// subtracting 1032 (72) leaves c - 8 exactly.  An integer of magnitude <= 8
// has at most 3 significant bits, so the low byte of its fp16 encoding is
// zero and the high byte is its e5m2 encoding (same exponent bias, 2
// mantissa bits): one byte permute packs four of them.
__device__ __forceinline__ uint2 e5m2_of_codes8(uint32_t w) {
  const uint32_t w8 = w >> 8;
  const __half2 lo_off = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  const __half2 hi_off = __halves2half2(__ushort_as_half(0x5480), __ushort_as_half(0x5480));
  uint32_t q[4] = {(w & 0x000F000Fu) | 0x64006400u, (w & 0x00F000F0u) | 0x54005400u,
                   (w8 & 0x000F000Fu) | 0x64006400u, (w8 & 0x00F000F0u) | 0x54005400u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&q[i]), (i & 1) ? hi_off : lo_off);
    q[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
  // q0 = (c0, c4), q1 = (c1, c5), q2 = (c2, c6), q3 = (c3, c7) as fp16 pairs:
  // high bytes 1 and 3 of each
  return make_uint2(prmt(q[0], q[1], 0x7351u), prmt(q[2], q[3], 0x7351u));
}

// Position of element i (0..7) of an aligned group of 8 in that order.
__device__ __forceinline__ int op_pos8(int i) { return (i & 1) | ((i & 2) << 1) | ((i & 4) >> 1); }

// D[tmem] = A[tmem] x B[smem]^T, kind::f8f6f4 (no accumulation into D: each
// scale group has an accumulator of its own).  A: 128 lanes (rows) x K = 32
// bytes in 8 consecutive columns, element k in byte k % 4 of column k / 4.
__device__ __forceinline__ void umma_f8_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc) {
  asm volatile("tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, 0;" ::"r"(d_tmem),
               "r"(a_tmem), "l"(b_desc), "r"(idesc)
               : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Scale of group g (0..7) from eight bf16 scales in a uint4.
__device__ __forceinline__ float scale_of(const uint4& v, int g) {
  const uint32_t w = g < 2 ? v.x : g < 4 ? v.y : g < 6 ? v.z : v.w;
  return (g & 1) ? bf16_hi(w) : bf16_lo(w);
}

// 32 TMEM lanes x W consecutive 32-bit columns (W = 2, 4, 8 or 16; see
// tmem_ld_32x32b_x16): the epilogue reads only the columns that hold tokens.
template <int W>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[W]) {
  if constexpr (W == 2) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"(taddr)
                 : "memory");
  } else if constexpr (W == 4) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr)
                 : "memory");
  } else if constexpr (W == 8) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr)
        : "memory");
  } else {
    static_assert(W == 16, "column count");
    tmem_ld_32x32b_x16(taddr, r);
  }
}

// Gate/up epilogue, one TMEM load batch: the accumulators of kGroupsPerLoad
// scale groups (gate at tq + 32 jj, up 16 columns further), W live columns
// each, scaled by the groups' scales and added into acc0 (gate) / acc1 (up).
template <int W>
__device__ __forceinline__ void gateup_batch(uint32_t tq, const uint4& s0, const uint4& s1,
                                             int gb, float (&acc0)[16], float (&acc1)[16]) {
  uint32_t v[kGroupsPerLoad][2][W];
#pragma unroll
  for (int jj = 0; jj < kGroupsPerLoad; ++jj) {
    tmem_ld_cols<W>(tq + jj * 32, v[jj][0]);
    tmem_ld_cols<W>(tq + jj * 32 + 16, v[jj][1]);
  }
  tmem_ld_wait();
#pragma unroll
  for (int jj = 0; jj < kGroupsPerLoad; ++jj) {
    const float sa = scale_of(s0, gb + jj), sb = scale_of(s1, gb + jj);
#pragma unroll
    for (int c = 0; c < W; ++c) {
      acc0[c] = fmaf(sa, __uint_as_float(v[jj][0][c]), acc0[c]);
      acc1[c] = fmaf(sb, __uint_as_float(v[jj][1][c]), acc1[c]);
    }
  }
}

// 4 x 4 transpose across the four lanes 4j .. 4j+3 of a warp: lane 4j+r
// holds row r, (x0, x1, x2, x3) = M[r][0..3], and ends with column r.
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

__device__ __forceinline__ uint8_t e4m3_rn(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float e4m3_value(uint8_t b) {
  return __half2float(__half(__nv_cvt_fp8_to_halfraw(b, __NV_E4M3)));
}

template <int NA, int EPI, bool kDown>
__global__ void __launch_bounds__(kThreads, 1)
    int4_f8_gemm_kernel(const __grid_constant__ CUtensorMap tm_c0,
                        const __grid_constant__ CUtensorMap tm_c1,
                        const __grid_constant__ CUtensorMap tm_sc0,
                        const __grid_constant__ CUtensorMap tm_sc1,
                        const __grid_constant__ CUtensorMap tm_b, const F8Args a) {
  using Cfg = F8Cfg<NA, kDown>;
  constexpr int P = Cfg::kPlanes;
  constexpr int kTok = Cfg::kMaxTok;
  // output rows per tile: two 128-row blocks for the paired down
  constexpr int kTileRows = (kDown && NA == 2) ? 2 * kBM : kBM;
  extern __shared__ uint8_t smem_raw[];
  // down: each epilogue warp's copy of its tile's h scales [token][group]
  __shared__ float s_hb[kDown ? 4 : 1][kDown ? kTok : 1][kDown ? kMaxGroups : 1];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* raws = base;
  uint8_t* bring = raws + Cfg::kRaw * Cfg::kRawBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(bring + kBStages * kBStageBytes);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + Cfg::kRaw;
  uint64_t* b_full = raw_empty + Cfg::kRaw;
  uint64_t* b_empty = b_full + kBStages;
  uint64_t* a_full = b_empty + kBStages;
  uint64_t* acc_full = a_full + Cfg::kSlots;
  uint64_t* acc_empty = acc_full + Cfg::kAccRing;
  uint64_t* drain = acc_empty + Cfg::kAccRing;  // one per issuer
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + kIssuers);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::kRaw; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], kDqThreads);
    }
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], kIssuers);
    }
    for (int i = 0; i < Cfg::kSlots; ++i) mbar_init(&a_full[i], kDqThreads);
    for (int i = 0; i < Cfg::kAccRing; ++i) {
      mbar_init(&acc_full[i], kIssuers);
      mbar_init(&acc_empty[i], 128);
    }
    for (int i = 0; i < kIssuers; ++i) mbar_init(&drain[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
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
  const int RB = a.K / kRawK;      // raw stages per tile (K % 256 == 0)
  const int KS = a.K / kSlotK;     // operand slots per tile
  const int G = a.K / 32;          // scale groups per tile

  auto code_tile = [&](int rs, int m) {
    return raws + rs * Cfg::kRawBytes + m * kCodeTileBytes;
  };
  // TMEM column of operand slot os, matrix m (lane 0)
  auto a_col = [&](int os, int m) {
    return static_cast<uint32_t>(Cfg::kABase + os * Cfg::kACols + m * kGroupsPerSlot * 8);
  };
  auto b_tile = [&](int bs, int sub) { return bring + bs * kBStageBytes + sub * kBTileBytes; };

  if (warp == 0) {
    // ---------------------------------------------------------------- code producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int rs = 0;
      uint32_t rph = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileEntry te = table_entry(a.table, tile / a.mblocks);
        const int mb = tile % a.mblocks;
        const bool sh = te.group == a.E;
        const int ge = sh ? 0 : te.group;
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
          if (NA == 2)  // the up matrix, or the down weights' second row block
            tma_load_3d(code_tile(rs, 1), sh ? &tm_sc1 : &tm_c1, &raw_full[rs], rb * (kRawK / 2),
                        kDown ? mb * kTileRows + kBM : mb * kBM, ge, pol);
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
      const uint64_t pol = policy_evict_last();
      int bs = 0;
      uint32_t bph = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileEntry te = table_entry(a.table, tile / a.mblocks);
        for (int k0 = 0; k0 < KS; k0 += kBSub) {
          const int nsub = min(kBSub, KS - k0);
          if (!mbar_wait(&b_empty[bs], bph ^ 1u, ab)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&b_full[bs], nsub * kBTileBytes);
          armed |= 1u << bs;
          armed_par = (armed_par & ~(1u << bs)) | (bph << bs);
          for (int sub = 0; sub < nsub; ++sub)
            tma_load_2d(b_tile(bs, sub), &tm_b, &b_full[bs], (k0 + sub) * kSlotK, P * te.row0,
                        pol);
          if (++bs == kBStages) {
            bs = 0;
            bph ^= 1u;
          }
        }
      }
      for (int s = 0; s < kBStages; ++s)
        if ((armed >> s) & 1u) mbar_wait_drain(&b_full[s], (armed_par >> s) & 1u);
    }
  } else if (warp >= 6 && warp < kDqWarpEnd) {
    // ---------------------------------------------------------------- dequantisers
    // a warp writes the TMEM lane quadrant (warp id % 4): row r of the tile
    // is lane r; warps 6..9 take one matrix (or the first two groups of a
    // slot), warps 10..13 the other
    const int dw = (threadIdx.x - kDqThread0) >> 5;  // 0..7
    const int r = (warp & 3) * 32 + lane;            // weight row of the tile = TMEM lane
    const int m = NA == 2 ? (dw >> 2) : 0;           // gate/up: matrix
    const int j0 = NA == 2 ? 0 : (dw >> 2) * 2;      // down: first of two groups per slot
    constexpr int kJ = NA == 2 ? kGroupsPerSlot : 2;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const int sw = r & 7;                       // 128-byte swizzle phase of this row
    int rs = 0, os = 0;
    uint32_t rph = 0;
    int n = 0;  // slots written so far (the MMA thread's accumulator entry n % kAccRing)
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      for (int rb = 0; ok && rb < RB; ++rb) {
        // warp-uniform waits: the TMEM stores below are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(&raw_full[rs], rph, ab))) {
          ok = false;
          break;
        }
        const uint8_t* ct = code_tile(rs, m) + r * 128;
#pragma unroll
        for (int sb = 0; sb < kSlotsPerRaw; ++sb) {
          // code chunk 4 sb + j (32 codes, one scale group) -> the group's 32
          // e5m2 bytes, TMEM columns 8 j .. 8 j + 7 of this row's lane
          uint32_t wv[kJ * 8];
#pragma unroll
          for (int jj = 0; jj < kJ; ++jj) {
            const int j = j0 + jj;
            const uint4 cw = *reinterpret_cast<const uint4*>(ct + (((sb * 4 + j) ^ sw) << 4));
            const uint2 e0 = e5m2_of_codes8(cw.x), e1 = e5m2_of_codes8(cw.y);
            const uint2 e2 = e5m2_of_codes8(cw.z), e3 = e5m2_of_codes8(cw.w);
            wv[8 * jj + 0] = e0.x;
            wv[8 * jj + 1] = e0.y;
            wv[8 * jj + 2] = e1.x;
            wv[8 * jj + 3] = e1.y;
            wv[8 * jj + 4] = e2.x;
            wv[8 * jj + 5] = e2.y;
            wv[8 * jj + 6] = e3.x;
            wv[8 * jj + 7] = e3.y;
          }
          // the MMAs of slot n - kSlots, the last to read these columns, have
          // completed: the commit of their accumulator entry has arrived
          if (n >= Cfg::kSlots) {
            const int p = n - Cfg::kSlots;
            if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[p % Cfg::kAccRing],
                                                   (p / Cfg::kAccRing) & 1, ab))) {
              ok = false;
              break;
            }
          }
          tc_fence_after_sync();
          const uint32_t tcol = lane_base + a_col(os, m) + j0 * 8;
          if constexpr (NA == 2)
            tmem_st_32x32b_x32(tcol, wv);
          else
            tmem_st_32x32b_x16(tcol, wv);
          tmem_st_wait();
          tc_fence_before_sync();
          mbar_arrive(&a_full[os]);
          ++n;
          if (++os == Cfg::kSlots) os = 0;
        }
        if (!ok) break;
        mbar_arrive(&raw_empty[rs]);
        if (++rs == Cfg::kRaw) {
          rs = 0;
          rph ^= 1u;
        }
      }
    }
  } else if (warp == 1 || warp == kMmaWarp1) {
    // ---------------------------------------------------------------- MMA issuers
    if (lane == 0) {
      const int mi = warp == 1 ? 0 : 1;  // issuer: matrix (gate/up) or group pair (down)
      // A e5m2 (format 1, bits 7..9), B e4m3 (format 0), fp32 accumulate
      const uint32_t idesc = idesc_f16(kBM, kBRows, false) | (1u << 7);
      // gate/up: all four groups of matrix mi; down: groups 2 mi, 2 mi + 1
      constexpr int kMyGroups = NA == 2 ? kGroupsPerSlot : kGroupsPerSlot / kIssuers;
      const int g0 = NA == 2 ? 0 : mi * kMyGroups;
      const uint32_t acc_off = NA == 2 ? mi * 16 : 0;  // gate / up accumulator of a group
      int os = 0, bs = 0, ring = 0;
      uint32_t oph = 0, bph = 0, rph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        for (int ks = 0; ks < KS; ++ks) {
          const int sub = ks % kBSub;
          if ((sub == 0 && !mbar_wait(&b_full[bs], bph, ab)) || !mbar_wait(&a_full[os], oph, ab) ||
              !mbar_wait(&acc_empty[ring], rph ^ 1u, ab)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t db = sw128_kmajor_desc(smem_u32(b_tile(bs, sub)));
          const uint32_t ta = tmem_base + a_col(os, NA == 2 ? mi : 0);
          const uint32_t dacc = tmem_base + ring * Cfg::kEntryCols + acc_off;
#pragma unroll
          for (int jj = 0; jj < kMyGroups; ++jj) {
            const int j = g0 + jj;
            umma_f8_tmem_a(dacc + j * Cfg::kGroupCols, ta + 8 * j, db + 2 * j, idesc);
          }
          umma_commit(&acc_full[ring]);
          if (++ring == Cfg::kAccRing) {
            ring = 0;
            rph ^= 1u;
          }
          if (++os == Cfg::kSlots) {
            os = 0;
            oph ^= 1u;
          }
          if (sub == kBSub - 1 || ks == KS - 1) {  // the stage's last slot
            umma_commit(&b_empty[bs]);
            if (++bs == kBStages) {
              bs = 0;
              bph ^= 1u;
            }
          }
        }
      }
      umma_commit(&drain[mi]);
      mbar_wait_drain(&drain[mi], 0);
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int q = warp & 3;
    const int r = q * 32 + lane;  // weight row of the tile = TMEM lane
    int ring = 0;
    uint32_t rph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      const TileEntry te = table_entry(a.table, tile / a.mblocks);
      const int mb = tile % a.mblocks;
      const bool sh = te.group == a.E;
      const int f = mb * kTileRows + r;  // output feature (N_out % 128 == 0)
      const int nt = min(te.nrows, kTok);
      const size_t srow = (static_cast<size_t>(sh ? 0 : te.group) * a.N_out + f) * G;
      // scales of the second matrix: up's row f, or the second block's row f + 128
      const size_t srow1 = srow + (kDown ? static_cast<size_t>(kBM) * G : 0);
      const uint4* s0p = reinterpret_cast<const uint4*>((sh ? a.sscale0 : a.scale0) + srow);
      const uint4* s1p = reinterpret_cast<const uint4*>((sh ? a.sscale1 : a.scale1) + srow1);
      // down, scatter-add: lane l < nt holds token l's id and routing weight
      int tk = -1;
      float tw = 0.f;
      if (kDown && EPI == kEpiScatterAdd && lane < nt && te.row0 + lane < a.total_rows) {
        const int t = a.gather[te.row0 + lane];
        tw = a.roww[te.row0 + lane];
        tk = (t >= 0 && t < a.out_rows) ? t : -1;
      }
      // gate/up: (gate, up) per B column; down: per token (and row block)
      constexpr int kAcc0 = kDown ? kTok : 16, kAcc1 = NA == 2 ? kAcc0 : 1;
      float acc0[kAcc0], acc1[kAcc1];
#pragma unroll
      for (int c = 0; c < kAcc0; ++c) acc0[c] = 0.f;
#pragma unroll
      for (int c = 0; c < kAcc1; ++c) acc1[c] = 0.f;
      if (kDown) {
        // the tile's h scales (1 / sigma) for every token and group, loaded
        // once into this warp's shared-memory copy (the warp's previous tile
        // is done with it: all lanes passed its group loop)
        __syncwarp();
        for (int i = lane; i < kTok * G; i += 32) {
          const int t = i / G, g = i - t * G;
          const int rr = te.row0 + t;
          s_hb[kDown ? q : 0][kDown ? t : 0][kDown ? g : 0] =
              (t < nt && rr < a.total_rows) ? __ldg(a.binv + static_cast<size_t>(rr) * G + g) : 0.f;
        }
        __syncwarp();
      }
      uint4 s0 = __ldg(s0p), s1 = NA == 2 ? __ldg(s1p) : s0;
      for (int g8 = 0; ok && g8 < G; g8 += 8) {
        // the next eight scales of each matrix, loaded one batch ahead
        const uint4 s0n = g8 + 8 < G ? __ldg(s0p + g8 / 8 + 1) : s0;
        const uint4 s1n = (NA == 2 && g8 + 8 < G) ? __ldg(s1p + g8 / 8 + 1) : s1;
#pragma unroll
        for (int gi = 0; gi < 8; gi += kGroupsPerSync) {
          if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[ring], rph, ab))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t tq0 =
              tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ring * Cfg::kEntryCols;
#pragma unroll
          for (int gl = 0; gl < kGroupsPerSync; gl += kGroupsPerLoad) {
            const uint32_t tq = tq0 + gl * Cfg::kGroupCols;
            const int gb = gi + gl;  // first group of this load batch within the eight
            if constexpr (!kDown) {
              // 2 nt live columns (hi and lo plane of each token)
              if (nt == 1)
                gateup_batch<2>(tq, s0, s1, gb, acc0, acc1);
              else if (nt <= 2)
                gateup_batch<4>(tq, s0, s1, gb, acc0, acc1);
              else if (nt <= 4)
                gateup_batch<8>(tq, s0, s1, gb, acc0, acc1);
              else
                gateup_batch<16>(tq, s0, s1, gb, acc0, acc1);
            } else {
              // 3 nt live columns (hi, mid and lo plane of each token); with
              // two row blocks the second block's accumulator is 16 columns on
              auto down_batch = [&](auto wtag) {
                constexpr int W = decltype(wtag)::value;
                constexpr int kT = W == 16 ? kTok : W / 3;
                constexpr int kGC = Cfg::kGroupCols;  // 16 or 32
                uint32_t v[kGroupsPerLoad][NA][W];
#pragma unroll
                for (int jj = 0; jj < kGroupsPerLoad; ++jj)
#pragma unroll
                  for (int m = 0; m < NA; ++m) tmem_ld_cols<W>(tq + jj * kGC + m * 16, v[jj][m]);
                tmem_ld_wait();
#pragma unroll
                for (int jj = 0; jj < kGroupsPerLoad; ++jj) {
                  const float sa = scale_of(s0, gb + jj);
                  [[maybe_unused]] const float sb = NA == 2 ? scale_of(s1, gb + jj) : 0.f;
#pragma unroll
                  for (int t = 0; t < kT; ++t) {
                    const float hbv = s_hb[kDown ? q : 0][kDown ? t : 0][kDown ? g8 + gb + jj : 0];
                    const float pv = (__uint_as_float(v[jj][0][3 * t]) +
                                      __uint_as_float(v[jj][0][3 * t + 1])) +
                                     __uint_as_float(v[jj][0][3 * t + 2]);
                    acc0[t] = fmaf(sa * hbv, pv, acc0[t]);
                    if constexpr (NA == 2) {
                      const float pv1 = (__uint_as_float(v[jj][1][3 * t]) +
                                         __uint_as_float(v[jj][1][3 * t + 1])) +
                                        __uint_as_float(v[jj][1][3 * t + 2]);
                      acc1[t] = fmaf(sb * hbv, pv1, acc1[t]);
                    }
                  }
                }
              };
              if (nt == 1)
                down_batch(std::integral_constant<int, 4>{});
              else if (nt <= 2)
                down_batch(std::integral_constant<int, 8>{});
              else
                down_batch(std::integral_constant<int, 16>{});
            }
          }
          tc_fence_before_sync();
          mbar_arrive(&acc_empty[ring]);
          if (++ring == Cfg::kAccRing) {
            ring = 0;
            rph ^= 1u;
          }
        }
        s0 = s0n;
        s1 = s1n;
      }
      if (!ok) break;
      if (!kDown) {
        // SwiGLU, then h as three e4m3 planes under a power-of-two scale per
        // (token, group of 32 features): the warp's 32 lanes are one group
        const int g32 = f >> 5;
        const int fpos = (f & ~7) | op_pos8(f & 7);
#pragma unroll
        for (int t = 0; t < kTok; ++t) {
          const int rr = te.row0 + t;
          if (t < nt && rr < a.total_rows) {  // the same for the whole warp
            const float inv = __ldg(a.binv + rr);
            const float gv = (acc0[2 * t] + acc0[2 * t + 1]) * inv;
            const float uv = (acc1[2 * t] + acc1[2 * t + 1]) * inv;
            const float hv = clamped_swiglu(gv, uv);
            float mx = fabsf(hv);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            int e = 0;
            if (mx > 0.f) frexpf(mx, &e);
            e = max(e, -100);
            const float sigma = ldexpf(1.0f, 8 - e);  // max |h sigma| in [128, 256)
            const float y = hv * sigma;
            const uint8_t b0 = e4m3_rn(y);
            const float r1 = y - e4m3_value(b0);
            const uint8_t b1 = e4m3_rn(r1);
            const uint8_t b2 = e4m3_rn(r1 - e4m3_value(b1));
            uint8_t* hp = a.h8 + static_cast<size_t>(rr) * 3 * a.N_out + fpos;
            hp[0] = b0;
            hp[a.N_out] = b1;
            hp[2 * a.N_out] = b2;
            if (lane == 0) a.hinv[static_cast<size_t>(rr) * (a.N_out / 32) + g32] = 1.0f / sigma;
          }
        }
      } else if (EPI == kEpiScatterAdd) {
        // lanes 4j .. 4j+3 hold four consecutive features: a 4 x 4 exchange
        // gives lane 4j+r those features of token tg + r, one 16-byte atomic
        // (two row blocks: the second block's features are 128 further on)
        const int r4 = lane & 3;
#pragma unroll
        for (int m = 0; m < NA; ++m) {
          float* const ob = a.out + ((f + m * kBM) & ~3);
#pragma unroll
          for (int tg = 0; tg < kTok; tg += 4) {
            float x[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int ti = (tg + i) % kTok;
              x[i] = tg + i < kTok ? (m == 0 ? acc0[ti] : acc1[NA == 2 ? ti : 0]) : 0.f;
            }
            transpose4_lanes(x[0], x[1], x[2], x[3], lane);
            const int t = tg + r4;
            const int tok = __shfl_sync(0xffffffffu, tk, t & 31);
            const float wr = __shfl_sync(0xffffffffu, tw, t & 31);
            if (t < nt && tok >= 0)
              atomicAdd(reinterpret_cast<float4*>(ob + static_cast<size_t>(tok) * a.N_out),
                        make_float4(wr * x[0], wr * x[1], wr * x[2], wr * x[3]));
          }
        }
      } else {
#pragma unroll
        for (int t = 0; t < kTok; ++t) {
          const int rr = te.row0 + t;
          if (t < nt && rr < a.total_rows) a.out[static_cast<size_t>(rr) * a.N_out + f] = acc0[t];
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int NA, int EPI, bool kDown>
cudaError_t f8_dispatch(const Int4F8Launch& L, cudaStream_t s) {
  using Cfg = F8Cfg<NA, kDown>;
  auto kern = int4_f8_gemm_kernel<NA, EPI, kDown>;
  constexpr int kTileRows = (kDown && NA == 2) ? 2 * kBM : kBM;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (err != cudaSuccess) return err;
  F8Args a{L.table, L.K, L.N_out, L.N_out / kTileRows, L.E, L.total_rows, L.out_rows,
           static_cast<const uint16_t*>(L.scale[0]), static_cast<const uint16_t*>(L.scale[1]),
           static_cast<const uint16_t*>(L.sscale[0]), static_cast<const uint16_t*>(L.sscale[1]),
           L.binv, L.h8, L.hinv, L.gather, L.roww, L.out, L.status, L.budget_ns};
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
  return cudaLaunchKernelEx(&cfg, kern, L.tm_c[0], L.tm_c[1], L.tm_sc[0], L.tm_sc[1], L.tm_b, a);
}

}  // namespace

cudaError_t launch_int4_f8_gemm(const Int4F8Launch& L, cudaStream_t s) {
  if (L.K % kRawK != 0 || L.N_out % kBM != 0) return cudaErrorInvalidValue;
  // down keeps the tile's h scales (K / 32 per token) in static shared memory
  // down (epilogue scatter-add or store rows; na = 2: two row blocks per
  // tile, scatter-add only) keeps the tile's h scales in static shared memory
  const bool down = L.epilogue != kEpiStoreRows || L.na == 1;
  if (down && L.K / 32 > kMaxGroups) return cudaErrorInvalidValue;
  if (L.na == 2 && L.epilogue == kEpiScatterAdd) {
    if (L.N_out % (2 * kBM) != 0) return cudaErrorInvalidValue;
    return f8_dispatch<2, kEpiScatterAdd, true>(L, s);
  }
  if (L.na == 2) return f8_dispatch<2, kEpiStoreRows, false>(L, s);
  if (L.epilogue == kEpiScatterAdd) return f8_dispatch<1, kEpiScatterAdd, true>(L, s);
  return f8_dispatch<1, kEpiStoreRows, true>(L, s);
}

}  // namespace moe
