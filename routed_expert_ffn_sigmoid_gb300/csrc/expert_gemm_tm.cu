// Token-major grouped expert GEMMs for large token counts (bf16 weights).
//
// Same per-expert computation as expert_gemm.cu (gate/up with the clamped
// SwiGLU; down with the routing weight and the scatter-add into the output;
// "Add GLM-5.3-Flash (glm5next) support with ROCmFP mix qtypes (105/106)",
// section "MoE FFN (REAL routed expert execution)"), oriented for groups of
// ~100+ tokens: the 128 token rows of a tile entry are the MMA's M operand
// and weight features are N (2 x 128 for gate/up, 256 for down).  Every MMA
// is full width, shared-memory operand bytes per flop drop by ~1.5x for the
// down projection, and the epilogue owns one token row per thread, so h is
// written with 16-byte stores and the output with 16-byte vector atomics.
//
// CTA = 7 warps (weight producer, MMA issuer, 4 epilogue warps, token
// producer), persistent over (tile-table entry, feature block) pairs,
// accumulators double-buffered in TMEM, every wait bounded as in the other
// GEMM kernels.  Weight tiles (from HBM) and token planes (mostly L2 hits)
// have rings of their own, so their depths are set apart: the down
// projection's two 16 KB token planes per K step no longer limit its weight
// ring to three stages (96 KB of HBM bytes in flight per SM; now 128 KB).
#include <cuda_bf16.h>

#include "moe_kernels.h"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;            // token rows per tile
constexpr int kBK = 64;
constexpr int kRowBytes = kBK * 2;  // 128
constexpr int kATileBytes = kBM * kRowBytes;  // 16 KB per token plane
constexpr int kThreads = 224;
constexpr int kGatherWarp = 6;    // token producer: TMA, or cp.async rows gathered from x

__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

// NA token planes (gate/up: x; down: h hi + lo), NBM weight matrices of
// FN features each (gate/up: 2 x 128; down: 1 x 256).
template <int NA, int NBM, int FN>
struct TmCfg {
  static constexpr int kBTileBytes = FN * kRowBytes;
  static constexpr int kAStageBytes = NA * kATileBytes;  // token planes of one K step
  static constexpr int kBStageBytes = NBM * kBTileBytes; // weight tiles of one K step
  // Measured at 1024-8192 tokens and on the dense FFN: gate/up is best with
  // 4 + 4 stages (fewer token stages, or a fifth weight stage, cost 10-35 %),
  // down with 3 + 4 (5-8 % faster than three shared stages of both).
  static constexpr int kAStages = NA == 2 ? 3 : 4;
  static constexpr int kBStages = 4;
  static constexpr int kAccCols = NBM * FN;  // 256 in both uses
  static constexpr int kAccStages = 2;
  static constexpr int kTmemCols = 512;
  static constexpr int kSmemBytes =
      kAStages * kAStageBytes + kBStages * kBStageBytes + 1024 + 256;
  static_assert(kAccStages * kAccCols <= 512, "TMEM");
  static_assert(NBM * FN <= 256, "one MMA spans every weight tile of a stage");
  static_assert(kAStageBytes % 1024 == 0 && kBStageBytes % 1024 == 0, "alignment");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kAStages + kBStages <= 16, "rings");
};

struct TmArgs {
  const int32_t* table;
  const int32_t* arows;   // gate/up: non-null -> token row r is xsrc[arows[r]] (cp.async)
  const uint16_t* xsrc;   // x [T][xpitch] bf16
  int xpitch;
  float4* zero_out;       // gate/up: cleared by the epilogue warps before their first tile
  size_t zero_n4;
  int K, N_out, nblocks, E, total_rows, out_rows;
  const int32_t* gather;
  const float* roww;
  float* out;
  void* h0;
  void* h1;
  int* status;
  uint64_t budget_ns;
};

__device__ __forceinline__ uint32_t pack_bf16x2(__nv_bfloat16 a, __nv_bfloat16 b) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(a)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
}

// EPI: kEpiStoreRows with NBM == 2 means the gate/up SwiGLU epilogue writing
// h (hi/lo bf16 planes); with NBM == 1, kEpiScatterAdd / kEpiStoreRows are the
// down epilogues.
template <int NA, int NBM, int FN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    tm_gemm_kernel(const __grid_constant__ CUtensorMap tm_a0,
                   const __grid_constant__ CUtensorMap tm_a1,
                   const __grid_constant__ CUtensorMap tm_b0,
                   const __grid_constant__ CUtensorMap tm_b1,
                   const __grid_constant__ CUtensorMap tm_sb0,
                   const __grid_constant__ CUtensorMap tm_sb1, const TmArgs a) {
  using Cfg = TmCfg<NA, NBM, FN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* aring = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* bring = aring + Cfg::kAStages * Cfg::kAStageBytes;
  uint64_t* a_full = reinterpret_cast<uint64_t*>(bring + Cfg::kBStages * Cfg::kBStageBytes);
  uint64_t* a_empty = a_full + Cfg::kAStages;
  uint64_t* b_full = a_empty + Cfg::kAStages;
  uint64_t* b_empty = b_full + Cfg::kBStages;
  uint64_t* tfull = b_empty + Cfg::kBStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // gathered token rows: each lane of the token producer warp arrives
  const bool gat = NA == 1 && a.arows != nullptr;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kAStages; ++s) {
      mbar_init(&a_full[s], gat ? 32 : 1);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < Cfg::kBStages; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
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
  const int total = a.table[0] * a.nblocks;
  const int KB = a.K / kBK;

  if (warp == 0) {
    // ---------------------------------------------------------------- weight producer
    if (lane == 0) {
      // weights read by one token tile stream through L2 (evict_first);
      // those of a group cut into several token tiles (the shared expert at
      // prefill, heavy experts) are read again by its other tiles
      const uint64_t pol_w = policy_evict_first(), pol_wr = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileEntry te = table_entry(a.table, tile / a.nblocks);
        const int nb = tile % a.nblocks;
        const bool sh = te.group == a.E;
        const int ge = sh ? 0 : te.group;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&b_empty[stage], phase ^ 1u, ab)) {
            ok = false;
            break;
          }
          uint8_t* sb = bring + stage * Cfg::kBStageBytes;
          mbar_arrive_expect_tx(&b_full[stage], Cfg::kBStageBytes);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          const uint64_t pw = te.ntiles > 1 ? pol_wr : pol_w;
          tma_load_3d(sb, sh ? &tm_sb0 : &tm_b0, &b_full[stage], kb * kBK, nb * FN, ge, pw);
          if (NBM == 2)
            tma_load_3d(sb + Cfg::kBTileBytes, sh ? &tm_sb1 : &tm_b1, &b_full[stage], kb * kBK,
                        nb * FN, ge, pw);
          if (++stage == Cfg::kBStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < Cfg::kBStages; ++s)
        if ((armed >> s) & 1u) mbar_wait_drain(&b_full[s], (armed_par >> s) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // gate/up: the gate and up tiles lie back to back in shared memory, so
      // one N = 256 MMA covers both (columns 0..127 gate, 128..255 up) and
      // reads each token tile once per K step instead of twice
      const uint32_t idesc = idesc_f16(kBM, NBM * FN, true);
      int sa = 0, sbs = 0, acc = 0;
      uint32_t pa = 0, pb = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, ab)) break;
        tc_fence_after_sync();
        const uint32_t d0 = tmem_base + acc * Cfg::kAccCols;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&b_full[sbs], pb, ab) || !mbar_wait(&a_full[sa], pa, ab)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t st = smem_u32(aring + sa * Cfg::kAStageBytes);
          const uint64_t da0 = sw128_kmajor_desc(st);
          const uint64_t da1 = sw128_kmajor_desc(st + kATileBytes);
          const uint64_t db0 = sw128_kmajor_desc(smem_u32(bring + sbs * Cfg::kBStageBytes));
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint32_t accum = (kb | k) != 0;
            umma_f16(d0, da0 + 2 * k, db0 + 2 * k, idesc, accum);
            if (NA == 2) umma_f16(d0, da1 + 2 * k, db0 + 2 * k, idesc, 1u);
          }
          umma_commit(&a_empty[sa]);
          umma_commit(&b_empty[sbs]);
          if (++sa == Cfg::kAStages) {
            sa = 0;
            pa ^= 1u;
          }
          if (++sbs == Cfg::kBStages) {
            sbs = 0;
            pb ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      umma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else if (warp == kGatherWarp) {
    if (!gat) {
      // ---------------------------------------------------------------- token producer (TMA)
      if (lane == 0) {
        // token planes: read by the nblocks tiles of their entry, which run
        // at about the same time; at prefill they exceed L2 (h is 9 T I 4
        // bytes), so they are not kept past that
        const uint64_t pol_x = policy_evict_normal();
        int stage = 0;
        uint32_t phase = 0, armed = 0, armed_par = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
          const TileEntry te = table_entry(a.table, tile / a.nblocks);
          for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait(&a_empty[stage], phase ^ 1u, ab)) {
              ok = false;
              break;
            }
            uint8_t* st = aring + stage * Cfg::kAStageBytes;
            mbar_arrive_expect_tx(&a_full[stage], Cfg::kAStageBytes);
            armed |= 1u << stage;
            armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
            tma_load_2d(st, &tm_a0, &a_full[stage], kb * kBK, te.row0, pol_x);
            if (NA == 2)
              tma_load_2d(st + kATileBytes, &tm_a1, &a_full[stage], kb * kBK, te.row0, pol_x);
            if (++stage == Cfg::kAStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        for (int s = 0; s < Cfg::kAStages; ++s)
          if ((armed >> s) & 1u) mbar_wait_drain(&a_full[s], (armed_par >> s) & 1u);
      }
    } else {
      // Token rows gathered from x by cp.async, in the stage order of the TMA
      // producer: eight lanes cover one 128-byte row (one 16-byte piece each,
      // placed in the 128-byte swizzle the MMA reads), so one instruction
      // copies four whole rows; rows past the group are left as they are
      // (they reach only output rows the epilogue never writes).  Up to
      // kDepth stages of copies stay in flight; for the oldest one every lane
      // waits for its copies, fences the async proxy and arrives.
      constexpr int kDepth = cmin(3, Cfg::kAStages);
      const int j = lane & 7;  // 16-byte piece of the row
      int stage = 0, inflight = 0;
      uint32_t phase = 0;
      bool ok = true;
      auto signal_oldest = [&]() {
        fence_proxy_async_smem();
        int so = stage - inflight;
        if (so < 0) so += Cfg::kAStages;
        mbar_arrive(&a_full[so]);
        --inflight;
      };
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileEntry te = table_entry(a.table, tile / a.nblocks);
        int tok[kBM / 4];  // token of row 4i + lane / 8
#pragma unroll
        for (int i = 0; i < kBM / 4; ++i) {
          const int r = 4 * i + (lane >> 3);
          tok[i] = r < te.nrows ? a.arows[te.row0 + r] : 0;
        }
        for (int kb = 0; kb < KB; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(&a_empty[stage], phase ^ 1u, ab))) {
            ok = false;
            break;
          }
          uint8_t* st = aring + stage * Cfg::kAStageBytes;
#pragma unroll
          for (int i = 0; i < kBM / 4; ++i) {
            const int r = 4 * i + (lane >> 3);
            if (r < te.nrows)
              cp_async_16(st + r * kRowBytes + ((j ^ (r & 7)) << 4),
                          a.xsrc + static_cast<size_t>(tok[i]) * a.xpitch + kb * kBK + j * 8);
          }
          cp_async_commit();
          ++inflight;
          if (++stage == Cfg::kAStages) {
            stage = 0;
            phase ^= 1u;
          }
          if (inflight == kDepth) {
            cp_async_wait<kDepth - 1>();
            signal_oldest();
          }
        }
      }
      cp_async_wait<0>();
      while (inflight > 0) signal_oldest();
    }
  } else {
    // The layer output is cleared here when asked (only the down GEMM, a
    // later launch, adds into it): the epilogue warps are otherwise idle
    // until their first accumulator is ready.
    if (a.zero_out) {
      const size_t nthr = static_cast<size_t>(gridDim.x) * 128;
      for (size_t i = static_cast<size_t>(blockIdx.x) * 128 + (threadIdx.x - 64); i < a.zero_n4; i += nthr)
        a.zero_out[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int q = warp & 3;
    const int lrow = q * 32 + lane;  // token row of the tile this thread owns
    // the scatter-add's output lines receive one addition per (token, slot)
    // spread over the launch: kept resident in L2 between them
    const uint64_t pol_out = policy_evict_last();
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const TileEntry te = table_entry(a.table, tile / a.nblocks);
      const int nb = tile % a.nblocks;
      // this thread's token id and weight, loaded while the tile's MMAs run
      const int r = te.row0 + lrow;
      const bool valid = lrow < te.nrows && r < a.total_rows;
      int t = 0;
      float wr = 0.f;
      if (EPI == kEpiScatterAdd && valid) {
        t = a.gather[r];
        wr = a.roww[r];
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, ab))) break;
      tc_fence_after_sync();
      const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * Cfg::kAccCols;
      const bool live = valid && (EPI != kEpiScatterAdd || (t >= 0 && t < a.out_rows));
      for (int c0 = 0; c0 < FN; c0 += 16) {
        uint32_t v0[16], v1[16];
        tmem_ld_32x32b_x16(tq + c0, v0);
        if (NBM == 2) tmem_ld_32x32b_x16(tq + FN + c0, v1);
        tmem_ld_wait();
        if (!live) continue;
        const int f = nb * FN + c0;  // first feature of this chunk
        if (NBM == 2) {
          uint32_t hi[8], lo[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float h0 = clamped_swiglu(__uint_as_float(v0[2 * i]), __uint_as_float(v1[2 * i]));
            const float h1 =
                clamped_swiglu(__uint_as_float(v0[2 * i + 1]), __uint_as_float(v1[2 * i + 1]));
            const __nv_bfloat16 a0 = __float2bfloat16_rn(h0), a1 = __float2bfloat16_rn(h1);
            hi[i] = pack_bf16x2(a0, a1);
            lo[i] = pack_bf16x2(__float2bfloat16_rn(h0 - __bfloat162float(a0)),
                                __float2bfloat16_rn(h1 - __bfloat162float(a1)));
          }
          uint4* ph = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.h0) +
                                               static_cast<size_t>(r) * a.N_out + f);
          uint4* pl = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.h1) +
                                               static_cast<size_t>(r) * a.N_out + f);
          ph[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          ph[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
          pl[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          pl[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
        } else if (EPI == kEpiScatterAdd) {
          float* po = a.out + static_cast<size_t>(t) * a.N_out + f;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            red_add_f32x4(po + 4 * i,
                          make_float4(wr * __uint_as_float(v0[4 * i]),
                                      wr * __uint_as_float(v0[4 * i + 1]),
                                      wr * __uint_as_float(v0[4 * i + 2]),
                                      wr * __uint_as_float(v0[4 * i + 3])),
                          pol_out);
        } else {
          float4* po = reinterpret_cast<float4*>(a.out + static_cast<size_t>(r) * a.N_out + f);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            po[i] = make_float4(__uint_as_float(v0[4 * i]), __uint_as_float(v0[4 * i + 1]),
                                __uint_as_float(v0[4 * i + 2]), __uint_as_float(v0[4 * i + 3]));
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

template <int NA, int NBM, int FN, int EPI>
cudaError_t tm_dispatch(const TmLaunch& L, cudaStream_t s) {
  using Cfg = TmCfg<NA, NBM, FN>;
  auto kern = tm_gemm_kernel<NA, NBM, FN, EPI>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (err != cudaSuccess) return err;
  TmArgs a{L.table, L.arows, static_cast<const uint16_t*>(L.xsrc), L.xpitch,
           reinterpret_cast<float4*>(L.zero_out), L.zero_out ? L.zero_n / 4 : 0, L.K, L.N_out, L.nblocks, L.E, L.total_rows, L.out_rows,
           L.gather, L.roww, L.out, L.h0, L.h1, L.status, L.budget_ns};
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
  return cudaLaunchKernelEx(&cfg, kern, L.tm_a[0], L.tm_a[1], L.tm_b[0], L.tm_b[1], L.tm_sb[0],
                            L.tm_sb[1], a);
}

}  // namespace

cudaError_t launch_tm_gemm(const TmLaunch& L, cudaStream_t s) {
  if (L.gateup) return tm_dispatch<1, 2, 128, kEpiStoreRows>(L, s);
  if (L.epilogue == kEpiScatterAdd) return tm_dispatch<2, 1, 256, kEpiScatterAdd>(L, s);
  return tm_dispatch<2, 1, 256, kEpiStoreRows>(L, s);
}

}  // namespace moe
