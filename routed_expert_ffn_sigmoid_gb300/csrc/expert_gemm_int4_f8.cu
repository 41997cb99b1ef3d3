// Grouped gate/up GEMM over grouped-Int4 weights on 8-bit tensor-core
// operands, for decode-size groups (at most 8 tokens per tile entry).
//
// Weights use the grouped fmt=4 Int4 format decoded as offset-binary,
// value = (nibble - 8) * scale ("feat(glm53): add device-resident HIP backend
// for MI350P", section "Key changes"), one bf16 scale per 32 reduction
// elements; gate/up and the clamped SwiGLU follow "Add GLM-5.3-Flash
// (glm5next) support with ROCmFP mix qtypes (105/106)", section "MoE FFN
// (REAL routed expert execution)".
//
// Why 8-bit operands.  With fp16 operand tiles the Int4 GEMM is bound by
// shared memory: per weight the dequantisers store 2 bytes and the tensor
// core reads 2 more.  Here the code n - 8 (an integer in [-8, 7], exact in
// e5m2) is the A operand, 1 byte per weight, and the scale is applied after
// the product:
//   sum_k (n_k - 8) s_g x_k = s_g * sum_{k in g} (n_k - 8) x_k,
// so each MMA covers exactly one scale group (K = 32 for kind::f8f6f4) into an
// accumulator of its own, and the epilogue warps add s_g times it into
// registers.  The token rows enter as two e4m3 planes under a power-of-two
// scale per row, hi = e4m3(x sigma) and lo = e4m3(x sigma - hi): bf16 has 8
// significant bits, hi holds the top 4 and the remainder fits lo's 4, so
// hi + lo = x sigma exactly except for values more than ~2^-14 below the row
// maximum (absolute error below 2^-17 of the maximum).  Every product is then
// exact in fp32, and only fp32 accumulation rounds, as in the fp16 path.
//
// B operand: rows 2t (hi) and 2t + 1 (lo) of token t, so N = 16 covers 8
// tokens; columns past the tile entry's rows are ignored.  Along K both
// operands hold each aligned group of 8 elements in the order
// (0, 1, 4, 5, 2, 3, 6, 7), the order the weight bytes come out of
// e5m2_of_codes8.
//
// CTA = 15 warps, persistent over the flat tile list:
//   warp 0, lane 0   code producer: TMA of packed codes, 256 reduction
//                    elements of both matrices per raw stage
//   warp 1           TMEM allocation; lane 0 issues tcgen05.mma kind::f8f6f4
//                    (A e5m2, B e4m3)
//   warps 2..5       epilogue: per scale group, tcgen05.ld of the group's
//                    accumulator, scale and add; after the last group the
//                    clamped SwiGLU and the fp16 h store
//   warps 6..13      dequantisers, one thread per (weight row, matrix): code
//                    words -> e5m2 bytes (fp16 mask-and-or, one half2
//                    subtract, one byte permute per four codes), written
//                    into the 128-byte-swizzled operand tile
//   warp 14, lane 0  token producer: TMA of the e4m3 token planes
// Accumulators: a ring of 8 entries of two groups x (16 gate + 16 up
// columns) = 512 TMEM columns; the MMA thread commits and the epilogue warps
// release one entry per two groups.  Every wait is bounded as in the other
// GEMM kernels.
#include <cuda_fp16.h>

#include "moe_kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;
constexpr int kSlotK = 128;                        // e4m3 per 128-byte swizzle row
constexpr int kRawK = 256;                         // reduction elements per raw stage
constexpr int kSlotsPerRaw = kRawK / kSlotK;       // 2
constexpr int kGroupsPerSlot = kSlotK / 32;        // 4
constexpr int kATileBytes = kBM * kSlotK;          // 16 KB e4m3 operand per matrix
constexpr int kSlotBytes = 2 * kATileBytes;        // gate + up
constexpr int kCodeTileBytes = kBM * (kRawK / 2);  // 16 KB packed codes per matrix
constexpr int kRawBytes = 2 * kCodeTileBytes;
constexpr int kBRows = 16;                         // hi/lo rows of up to 8 tokens
constexpr int kBTileBytes = kBRows * kSlotK;       // 2 KB
constexpr int kRaw = 4;
constexpr int kSlots = 2;
constexpr int kBStages = 8;
constexpr int kGroupsPerSync = 2;                  // groups per accumulator handshake
constexpr int kAccRing = 8;                        // handshakes in flight (16 groups)
constexpr int kAccCols = 32 * kGroupsPerSync;      // per group: 16 gate + 16 up columns
constexpr int kTmemCols = kAccRing * kAccCols;     // 512
constexpr int kBarBytes = 1024;
constexpr int kSmemBytes =
    kSlots * kSlotBytes + kRaw * kRawBytes + kBStages * kBTileBytes + 1024 + kBarBytes;
constexpr int kThreads = 480;
constexpr int kDqThread0 = 192;
constexpr int kDqThreads = 256;
constexpr int kDqWarpEnd = 14;
constexpr int kBWarp = 14;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
static_assert(kTmemCols == 512, "TMEM");

struct F8Args {
  const int32_t* table;
  int K, N_out, mblocks, E, total_rows;
  const uint16_t* gate_scale;   // routed scales [E][N_out][K / 32] bf16
  const uint16_t* up_scale;
  const uint16_t* sgate_scale;  // shared expert [1][N_out][K / 32]
  const uint16_t* sup_scale;
  const float* xinv;            // per token row: 1 / sigma
  __half* h;                    // [rows][N_out], columns in the Int4 operand order
  int* status;
  uint64_t budget_ns;
};

__device__ __forceinline__ TileEntry entry_at(const int32_t* table, int i) {
  const int4 v =
      reinterpret_cast<const int4*>(reinterpret_cast<const char*>(table) + kTableHeaderBytes)[i];
  return TileEntry{v.x, v.y, v.z, v.w};
}

__device__ __forceinline__ float clamped_swiglu(float g, float u) {
  const float gc = fminf(g, 10.0f);
  const float uc = fminf(fmaxf(u, -10.0f), 10.0f);
  return gc / (1.0f + expf(-gc)) * uc;
}

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

__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 TMEM lanes x 8 consecutive 32-bit columns (see tmem_ld_32x32b_x16).
__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Scale of group g (0..7) from eight bf16 scales in a uint4.
__device__ __forceinline__ float scale_of(const uint4& v, int g) {
  const uint32_t w = g < 2 ? v.x : g < 4 ? v.y : g < 6 ? v.z : v.w;
  return (g & 1) ? bf16_hi(w) : bf16_lo(w);
}

__global__ void __launch_bounds__(kThreads, 1)
    int4_f8_gateup_kernel(const __grid_constant__ CUtensorMap tm_c0,
                          const __grid_constant__ CUtensorMap tm_c1,
                          const __grid_constant__ CUtensorMap tm_sc0,
                          const __grid_constant__ CUtensorMap tm_sc1,
                          const __grid_constant__ CUtensorMap tm_b, const F8Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* slots = base;
  uint8_t* raws = slots + kSlots * kSlotBytes;
  uint8_t* bring = raws + kRaw * kRawBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(bring + kBStages * kBTileBytes);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + kRaw;
  uint64_t* b_full = raw_empty + kRaw;
  uint64_t* b_empty = b_full + kBStages;
  uint64_t* a_full = b_empty + kBStages;
  uint64_t* op_empty = a_full + kSlots;
  uint64_t* acc_full = op_empty + kSlots;
  uint64_t* acc_empty = acc_full + kAccRing;
  uint64_t* drain = acc_empty + kAccRing;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRaw; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], kDqThreads);
    }
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&a_full[i], kDqThreads);
      mbar_init(&op_empty[i], 1);
    }
    for (int i = 0; i < kAccRing; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 128);
    }
    mbar_init(drain, 1);
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

  auto code_tile = [&](int rs, int m) { return raws + rs * kRawBytes + m * kCodeTileBytes; };
  auto a_tile = [&](int os, int m) { return slots + os * kSlotBytes + m * kATileBytes; };
  auto b_tile = [&](int bs) { return bring + bs * kBTileBytes; };

  if (warp == 0) {
    // ---------------------------------------------------------------- code producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int rs = 0;
      uint32_t rph = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileEntry te = entry_at(a.table, tile / a.mblocks);
        const int mb = tile % a.mblocks;
        const bool sh = te.group == a.E;
        const int ge = sh ? 0 : te.group;
        for (int rb = 0; rb < RB; ++rb) {
          if (!mbar_wait(&raw_empty[rs], rph ^ 1u, ab)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&raw_full[rs], kRawBytes);
          armed |= 1u << rs;
          armed_par = (armed_par & ~(1u << rs)) | (rph << rs);
          tma_load_3d(code_tile(rs, 0), sh ? &tm_sc0 : &tm_c0, &raw_full[rs], rb * (kRawK / 2),
                      mb * kBM, ge, pol);
          tma_load_3d(code_tile(rs, 1), sh ? &tm_sc1 : &tm_c1, &raw_full[rs], rb * (kRawK / 2),
                      mb * kBM, ge, pol);
          if (++rs == kRaw) {
            rs = 0;
            rph ^= 1u;
          }
        }
      }
      for (int s = 0; s < kRaw; ++s)
        if ((armed >> s) & 1u) mbar_wait_drain(&raw_full[s], (armed_par >> s) & 1u);
    }
  } else if (warp == kBWarp) {
    // ---------------------------------------------------------------- token producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();
      int bs = 0;
      uint32_t bph = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileEntry te = entry_at(a.table, tile / a.mblocks);
        for (int ks = 0; ks < KS; ++ks) {
          if (!mbar_wait(&b_empty[bs], bph ^ 1u, ab)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&b_full[bs], kBTileBytes);
          armed |= 1u << bs;
          armed_par = (armed_par & ~(1u << bs)) | (bph << bs);
          tma_load_2d(b_tile(bs), &tm_b, &b_full[bs], ks * kSlotK, 2 * te.row0, pol);
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
    const int d = threadIdx.x - kDqThread0;
    const int r = d & (kBM - 1);  // weight row of the tile
    const int m = d >> 7;         // matrix: 0 gate, 1 up
    const int sw = r & 7;         // 128-byte swizzle phase of this row
    int rs = 0, os = 0;
    uint32_t rph = 0, oph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      for (int rb = 0; ok && rb < RB; ++rb) {
        if (!mbar_wait(&raw_full[rs], rph, ab)) {
          ok = false;
          break;
        }
        const uint8_t* ct = code_tile(rs, m) + r * 128;
#pragma unroll
        for (int sb = 0; sb < kSlotsPerRaw; ++sb) {
          if (!mbar_wait(&op_empty[os], oph ^ 1u, ab)) {
            ok = false;
            break;
          }
          uint8_t* at = a_tile(os, m) + r * 128;
          // 128 codes of this slot: code chunks 4 sb .. 4 sb + 3 (32 codes,
          // one scale group each) -> e4m3 chunks 8 j' .. : chunk 2 j (+1)
          // holds codes 32 j .. 32 j + 15 (+16).
#pragma unroll
          for (int j = 0; j < kGroupsPerSlot; ++j) {
            const uint4 cw = *reinterpret_cast<const uint4*>(ct + (((sb * 4 + j) ^ sw) << 4));
            const uint2 e0 = e5m2_of_codes8(cw.x), e1 = e5m2_of_codes8(cw.y);
            const uint2 e2 = e5m2_of_codes8(cw.z), e3 = e5m2_of_codes8(cw.w);
            const uint4 o0 = make_uint4(e0.x, e0.y, e1.x, e1.y);
            const uint4 o1 = make_uint4(e2.x, e2.y, e3.x, e3.y);
            *reinterpret_cast<uint4*>(at + (((2 * j) ^ sw) << 4)) = o0;
            *reinterpret_cast<uint4*>(at + (((2 * j + 1) ^ sw) << 4)) = o1;
          }
          fence_proxy_async_smem();
          mbar_arrive(&a_full[os]);
          if (++os == kSlots) {
            os = 0;
            oph ^= 1u;
          }
        }
        if (!ok) break;
        mbar_arrive(&raw_empty[rs]);
        if (++rs == kRaw) {
          rs = 0;
          rph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      // A e5m2 (format 1, bits 7..9), B e4m3 (format 0), fp32 accumulate
      const uint32_t idesc = idesc_f16(kBM, kBRows, false) | (1u << 7);
      int os = 0, bs = 0, ring = 0;
      uint32_t oph = 0, bph = 0, rph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        for (int ks = 0; ks < KS; ++ks) {
          if (!mbar_wait(&b_full[bs], bph, ab) || !mbar_wait(&a_full[os], oph, ab)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t db = sw128_kmajor_desc(smem_u32(b_tile(bs)));
          const uint64_t dg = sw128_kmajor_desc(smem_u32(a_tile(os, 0)));
          const uint64_t du = sw128_kmajor_desc(smem_u32(a_tile(os, 1)));
#pragma unroll
          for (int j0 = 0; j0 < kGroupsPerSlot; j0 += kGroupsPerSync) {
            if (!mbar_wait(&acc_empty[ring], rph ^ 1u, ab)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
#pragma unroll
            for (int jj = 0; jj < kGroupsPerSync; ++jj) {
              const int j = j0 + jj;
              const uint32_t dacc = tmem_base + ring * kAccCols + jj * 32;
              umma_f8(dacc, dg + 2 * j, db + 2 * j, idesc, 0u);
              umma_f8(dacc + 16, du + 2 * j, db + 2 * j, idesc, 0u);
            }
            umma_commit(&acc_full[ring]);
            if (++ring == kAccRing) {
              ring = 0;
              rph ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit(&op_empty[os]);
          umma_commit(&b_empty[bs]);
          if (++os == kSlots) {
            os = 0;
            oph ^= 1u;
          }
          if (++bs == kBStages) {
            bs = 0;
            bph ^= 1u;
          }
        }
      }
      umma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int q = warp & 3;
    const int r = q * 32 + lane;  // weight row of the tile = TMEM lane
    int ring = 0;
    uint32_t rph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      const TileEntry te = entry_at(a.table, tile / a.mblocks);
      const int mb = tile % a.mblocks;
      const bool sh = te.group == a.E;
      const int f = mb * kBM + r;  // feature (N_out % 128 == 0)
      const size_t srow = (static_cast<size_t>(sh ? 0 : te.group) * a.N_out + f) * G;
      const uint4* sgp = reinterpret_cast<const uint4*>((sh ? a.sgate_scale : a.gate_scale) + srow);
      const uint4* sup = reinterpret_cast<const uint4*>((sh ? a.sup_scale : a.up_scale) + srow);
      const int live = 2 * te.nrows;  // accumulator columns that hold tokens
      float ag[16], au[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) ag[c] = au[c] = 0.f;
      uint4 sg = __ldg(sgp), su = __ldg(sup);
      for (int g8 = 0; ok && g8 < G; g8 += 8) {
        // the next eight scales of each matrix, loaded one batch ahead
        const uint4 sgn = g8 + 8 < G ? __ldg(sgp + g8 / 8 + 1) : sg;
        const uint4 sun = g8 + 8 < G ? __ldg(sup + g8 / 8 + 1) : su;
#pragma unroll
        for (int gi = 0; gi < 8; gi += kGroupsPerSync) {
          if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[ring], rph, ab))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ring * kAccCols;
          if (live <= 8) {
            // at most 4 tokens: columns 0..7 of each accumulator
            uint32_t v[kGroupsPerSync][2][8];
#pragma unroll
            for (int jj = 0; jj < kGroupsPerSync; ++jj) {
              tmem_ld_32x32b_x8(tq + jj * 32, v[jj][0]);
              tmem_ld_32x32b_x8(tq + jj * 32 + 16, v[jj][1]);
            }
            tmem_ld_wait();
            tc_fence_before_sync();
            mbar_arrive(&acc_empty[ring]);
#pragma unroll
            for (int jj = 0; jj < kGroupsPerSync; ++jj) {
              const float s_g = scale_of(sg, gi + jj), s_u = scale_of(su, gi + jj);
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                ag[c] = fmaf(s_g, __uint_as_float(v[jj][0][c]), ag[c]);
                au[c] = fmaf(s_u, __uint_as_float(v[jj][1][c]), au[c]);
              }
            }
          } else {
            uint32_t v[kGroupsPerSync][2][16];
#pragma unroll
            for (int jj = 0; jj < kGroupsPerSync; ++jj) {
              tmem_ld_32x32b_x16(tq + jj * 32, v[jj][0]);
              tmem_ld_32x32b_x16(tq + jj * 32 + 16, v[jj][1]);
            }
            tmem_ld_wait();
            tc_fence_before_sync();
            mbar_arrive(&acc_empty[ring]);
#pragma unroll
            for (int jj = 0; jj < kGroupsPerSync; ++jj) {
              const float s_g = scale_of(sg, gi + jj), s_u = scale_of(su, gi + jj);
#pragma unroll
              for (int c = 0; c < 16; ++c) {
                ag[c] = fmaf(s_g, __uint_as_float(v[jj][0][c]), ag[c]);
                au[c] = fmaf(s_u, __uint_as_float(v[jj][1][c]), au[c]);
              }
            }
          }
          if (++ring == kAccRing) {
            ring = 0;
            rph ^= 1u;
          }
        }
        sg = sgn;
        su = sun;
      }
      if (!ok) break;
      // column of feature f in the down GEMM's operand order (see expert_gemm_int4.cu)
      const int f_op = (f & ~7) | ((f & 3) << 1) | ((f >> 2) & 1);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int rr = te.row0 + t;
        if (t < te.nrows && rr < a.total_rows) {
          const float inv = __ldg(a.xinv + rr);
          const float gv = (ag[2 * t] + ag[2 * t + 1]) * inv;
          const float uv = (au[2 * t] + au[2 * t + 1]) * inv;
          a.h[static_cast<size_t>(rr) * a.N_out + f_op] = __float2half_rn(clamped_swiglu(gv, uv));
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

}  // namespace

cudaError_t launch_int4_f8_gateup(const Int4F8Launch& L, cudaStream_t s) {
  if (L.K % kRawK != 0 || L.N_out % kBM != 0) return cudaErrorInvalidValue;
  auto kern = int4_f8_gateup_kernel;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (err != cudaSuccess) return err;
  F8Args a{L.table, L.K, L.N_out, L.N_out / kBM, L.E, L.total_rows,
           static_cast<const uint16_t*>(L.gate_scale), static_cast<const uint16_t*>(L.up_scale),
           static_cast<const uint16_t*>(L.sgate_scale), static_cast<const uint16_t*>(L.sup_scale),
           L.xinv, static_cast<__half*>(L.h), L.status, L.budget_ns};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, L.tm_c[0], L.tm_c[1], L.tm_sc[0], L.tm_sc[1], L.tm_b, a);
}

}  // namespace moe
