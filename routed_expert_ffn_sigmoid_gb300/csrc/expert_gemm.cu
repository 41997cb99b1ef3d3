// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// operands streamed by TMA through an mbarrier ring.
//
// Per-expert gate / up / down matmuls ("ggml_mul_mat_id" for gate, up and
// down; clamped SwiGLU between gate/up and down; shared expert combined with
// the routed output -- "Add GLM-5.3-Flash (glm5next) support with ROCmFP mix
// qtypes (105/106)", section "MoE FFN (REAL routed expert execution)").
//
// Orientation ("swap AB"): the weight rows are the M = 128 operand and the
// tokens of one expert group are the N operand (16..256, chosen per tile), so
// a group of a few decode tokens still issues full-height MMAs and each
// weight byte crosses HBM once.  D[feature][token] accumulates in TMEM.
//
// CTA = 6 warps, persistent over a flat tile list:
//   warp 0, lane 0  TMA producer (weights evict-first, activations evict-last)
//   warp 1          TMEM allocation; lane 0 issues tcgen05.mma, commits
//   warps 2..5      epilogue: tcgen05.ld of their 32-lane TMEM quadrant
// Accumulators are double-buffered in TMEM where they fit, so the epilogue of
// one tile overlaps the main loop of the next.
//
// Every wait is bounded (AbortState): on a timeout the CTA records
// MOE_ERR_TIMEOUT in the workspace status word, drains the copies and MMAs it
// issued, frees TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_kernels.h"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;                      // MMA M: weight rows per tile
constexpr int kBK = 64;                       // K per stage: one 128-byte swizzle row
constexpr int kRowBytes = kBK * 2;            // 128
constexpr int kChunkRows = 16;                // token rows per activation TMA box
constexpr int kChunkBytes = kChunkRows * kRowBytes;
constexpr int kATileBytes = kBM * kRowBytes;  // 16 KB
constexpr int kStageBudget = 224 * 1024;
constexpr int kThreads = 192;

constexpr int ceil_pow2_32(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}
constexpr int cmin(int a, int b) { return a < b ? a : b; }

template <int BN>
struct GateUpCfg {
  static constexpr int kBTileBytes = BN * kRowBytes;
  static constexpr int kStageBytes = 2 * kATileBytes + kBTileBytes;
  static constexpr int kStages = cmin(8, kStageBudget / kStageBytes);
  static constexpr int kAccStages = (4 * BN <= 512) ? 2 : 1;
  static constexpr int kAccCols = 2 * BN;  // gate accumulator, then up accumulator
  static constexpr int kTmemCols = ceil_pow2_32(kAccStages * kAccCols);
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256;
  static_assert(kStageBytes % 1024 == 0, "stage tiles must stay 1024-byte aligned");
};

template <int BN, int NB>
struct DownCfg {
  static constexpr int kBTileBytes = BN * kRowBytes;
  static constexpr int kStageBytes = kATileBytes + NB * kBTileBytes;
  static constexpr int kStages = cmin(8, kStageBudget / kStageBytes);
  static constexpr int kAccStages = (2 * BN <= 512) ? 2 : 1;
  static constexpr int kTmemCols = ceil_pow2_32(kAccStages * BN);
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256;
  static_assert(kStageBytes % 1024 == 0, "stage tiles must stay 1024-byte aligned");
};

struct GateUpArgs {
  const int32_t* table;
  const int32_t* xrows;  // non-null: token rows gathered from x by xrows[r] (tm_x over x)
  int K, I, E, a_rows, total_rows;
  // > 0: the shared expert's first: its n_sh = ceil(T / BN) entries (rows
  // sh_row0 + t, token rows x[t] through tm_xs) lead the unit order and are
  // computed before the wait on the routing; the table's routed entries follow
  int n_sh, T, sh_row0;
  int ksplit;            // units per tile along K (1: no split)
  float* partial;        // ksplit > 1: fp32 partial G/U per unit
  int* counters;         // ksplit > 1: finished units per tile (zero between calls)
  void* h0;
  void* h1;
  int* status;
  uint64_t budget_ns;
};

struct DownArgs {
  const int32_t* table;
  int dense_rows;
  int ksplit;            // units per tile along K (scatter-add epilogue only)
  int K, N_out, mblocks, E, a_rows, total_rows, out_rows;
  const int32_t* gather;
  const float* roww;
  const float* bias;
  float* out;
  int* status;
  uint64_t budget_ns;
};

__device__ __forceinline__ int n_entries_of(const int32_t* table, int dense_rows, int BN) {
  return table ? table[0] : (dense_rows + BN - 1) / BN;
}

__device__ __forceinline__ TileEntry entry_at(const int32_t* table, int dense_rows, int BN, int i) {
  if (table) return table_entry(table, i);
  return TileEntry{0, i * BN, min(BN, dense_rows - i * BN), (dense_rows + BN - 1) / BN};
}

constexpr int kEpiThread0 = 64;  // first epilogue thread (warp 2)

// Barrier among the four epilogue warps only.
__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }


struct SmemCarve {
  uint8_t* tiles;
  uint64_t *full, *empty, *tfull, *tempty, *drain;
  uint32_t* tmem_holder;
  int* abort_flag;
  int* split_flags;  // [0]: an epilogue warp gave up, [1]: this unit finishes its tile
};

__device__ __forceinline__ SmemCarve carve(uint8_t* raw, int stages, int stage_bytes) {
  SmemCarve c;
  c.tiles = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  c.full = reinterpret_cast<uint64_t*>(c.tiles + stages * stage_bytes);
  c.empty = c.full + stages;
  c.tfull = c.empty + stages;
  c.tempty = c.tfull + 2;
  c.drain = c.tempty + 2;
  c.tmem_holder = reinterpret_cast<uint32_t*>(c.drain + 1);
  c.abort_flag = reinterpret_cast<int*>(c.tmem_holder + 1);
  c.split_flags = c.abort_flag + 1;
  return c;
}

__device__ __forceinline__ void init_barriers(const SmemCarve& c, int stages) {
  for (int s = 0; s < stages; ++s) {
    mbar_init(&c.full[s], 1);
    mbar_init(&c.empty[s], 1);
  }
  for (int i = 0; i < 2; ++i) {
    mbar_init(&c.tfull[i], 1);
    mbar_init(&c.tempty[i], 128);
  }
  mbar_init(c.drain, 1);
  *c.abort_flag = 0;
  c.split_flags[0] = 0;
  c.split_flags[1] = 0;
  fence_barrier_init();
}

// ======================================================================
// gate/up: D_g = W_gate[e] x X^T, D_u = W_up[e] x X^T, then the clamped
// SwiGLU.  bf16 path: h is stored as a hi/lo pair of bf16 planes (h = hi +
// lo to ~16 bits), which keeps the down projection's input error far below
// a bf16 rounding while the down MMA still takes bf16 operands.  fp16 path
// (Int4 weights): h is stored as one fp16 plane.
// ======================================================================
template <int BN, bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
    gateup_kernel(const __grid_constant__ CUtensorMap tm_gate,
                  const __grid_constant__ CUtensorMap tm_up,
                  const __grid_constant__ CUtensorMap tm_sgate,
                  const __grid_constant__ CUtensorMap tm_sup,
                  const __grid_constant__ CUtensorMap tm_x,
                  const __grid_constant__ CUtensorMap tm_xs, const GateUpArgs a) {
  using Cfg = GateUpCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  const SmemCarve sm = carve(smem_raw, Cfg::kStages, Cfg::kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    init_barriers(sm, Cfg::kStages);
    tma_prefetch_desc(&tm_gate);
    tma_prefetch_desc(&tm_up);
    tma_prefetch_desc(&tm_sgate);
    tma_prefetch_desc(&tm_sup);
    tma_prefetch_desc(&tm_x);
    if (a.n_sh) tma_prefetch_desc(&tm_xs);
  }
  if (warp == 1) {
    tmem_alloc(sm.tmem_holder, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *sm.tmem_holder;
  const AbortState ab{sm.abort_flag, a.status, a.budget_ns};

  pdl_launch_dependents();
  const int mblocks = (a.I + kBM - 1) / kBM;
  const int KB = a.K / kBK;
  // The shared expert's units need nothing the routing writes (its rows are
  // the tokens in order, read from x), so each role runs them before it
  // waits for the preceding kernels; the rest of the unit list comes from
  // the table after that wait.  Every role walks the same unit sequence.
  const int units_sh = a.n_sh * mblocks * a.ksplit;
  auto entry_of = [&](int i) -> TileEntry {
    if (i < a.n_sh)
      return TileEntry{a.E, a.sh_row0 + i * BN, min(BN, a.T - i * BN), a.n_sh};
    return entry_at(a.table, 0, BN, i - a.n_sh);
  };
  auto all_units = [&]() { return n_entries_of(a.table, 0, BN) * mblocks * a.ksplit; };
  // units this role may process so far; a role past them waits, then reads
  // the table (the routed entries plus the shared ones it already ran)
  auto advance = [&](int u, int& units, bool& waited) {
    if (u < units) return true;
    if (waited) return false;
    pdl_wait();
    waited = true;
    units = all_units();
    return u < units;
  };

  if (warp == 0) {
    // Producer warp.  Lane 0 waits for a free stage, arms it and loads the
    // weight tiles; the token rows come either as 16-row boxes of x_perm
    // (lane 0) or, with a.xrows, straight from x: lane L gathers rows
    // 4L .. 4L+3 of the tile (tile::gather4), so no permuted copy of x exists.
    // Only the tile's own rows are gathered (rounded up to 4); the rest of
    // the 16-row MMA block keeps whatever an earlier stage left there, which
    // reaches only output columns the epilogue never reads.
    const bool gat = a.xrows != nullptr;
    if (gat || lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_par = 0;
      bool ok = true;
      // A unit's table entry and gathered row indices are loaded one unit
      // ahead: between two units the producer never waits on a global load,
      // so the weight stream keeps its copies in flight.
      TileEntry te_next{};
      int tok_next[4] = {0, 0, 0, 0};
      int fetched = -1;  // unit whose entry / rows te_next, tok_next hold
      auto fetch_unit = [&](int uu) {
        const int ei = (uu / a.ksplit) / mblocks;
        te_next = entry_of(ei);
        if (gat && ei >= a.n_sh && lane < (te_next.nrows + 3) / 4) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tok_next[j] = a.xrows[te_next.row0 + min(4 * lane + j, te_next.nrows - 1)];
        }
        fetched = uu;
      };
      int units = a.n_sh ? units_sh : 0;
      bool waited = false;
      for (int u = blockIdx.x; ok && advance(u, units, waited); u += gridDim.x) {
        if (fetched != u) fetch_unit(u);
        const int tile = u / a.ksplit, sp = u % a.ksplit;
        const int kb0 = sp * KB / a.ksplit, kb1 = (sp + 1) * KB / a.ksplit;
        const TileEntry te = te_next;
        // gathered rows of this lane (rows past the group repeat its last row)
        const int tok[4] = {tok_next[0], tok_next[1], tok_next[2], tok_next[3]};
        // the next unit's entry ahead of time, while it needs no wait
        if (u + static_cast<int>(gridDim.x) < units) fetch_unit(u + gridDim.x);
        const bool shared_early = (tile / mblocks) < a.n_sh;  // rows straight from x (tm_xs)
        const int mb = tile % mblocks;
        const bool sh = te.group == a.E;
        const CUtensorMap* mg = sh ? &tm_sgate : &tm_gate;
        const CUtensorMap* mu = sh ? &tm_sup : &tm_up;
        const int ge = sh ? 0 : te.group;
        const int nchunks = (te.nrows + kChunkRows - 1) / kChunkRows;
        const int ngather = (te.nrows + 3) / 4;  // gather4 loads of the tile (gathered rows)
        const bool gat_u = gat && !shared_early;
        const uint32_t bytes = 2u * a.a_rows * kRowBytes +
                               (gat_u ? ngather * 4 * kRowBytes : nchunks * kChunkBytes);
        const bool issuer = gat_u && lane < ngather;
        for (int kb = kb0; kb < kb1; ++kb) {
          uint8_t* st = sm.tiles + stage * Cfg::kStageBytes;
          bool go = true;
          if (lane == 0) {
            go = mbar_wait(&sm.empty[stage], phase ^ 1u, ab);
            if (go) {
              mbar_arrive_expect_tx(&sm.full[stage], bytes);
              armed |= 1u << stage;
              armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
              tma_load_3d(st, mg, &sm.full[stage], kb * kBK, mb * kBM, ge, pol_w);
              tma_load_3d(st + kATileBytes, mu, &sm.full[stage], kb * kBK, mb * kBM, ge, pol_w);
              if (shared_early)
                for (int c = 0; c < nchunks; ++c)
                  tma_load_2d(st + 2 * kATileBytes + c * kChunkBytes, &tm_xs, &sm.full[stage],
                              kb * kBK, te.row0 - a.sh_row0 + c * kChunkRows, pol_x);
              else if (!gat)
                for (int c = 0; c < nchunks; ++c)
                  tma_load_2d(st + 2 * kATileBytes + c * kChunkBytes, &tm_x, &sm.full[stage],
                              kb * kBK, te.row0 + c * kChunkRows, pol_x);
            }
          }
          if (gat) go = __shfl_sync(0xffffffffu, go, 0);
          if (!go) {
            ok = false;
            break;
          }
          if (issuer)
            tma_gather4_2d(st + 2 * kATileBytes + lane * 4 * kRowBytes, &tm_x, &sm.full[stage],
                           kb * kBK, tok[0], tok[1], tok[2], tok[3], pol_x);
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every copy issued has landed before the CTA may exit
      if (lane == 0)
        for (int s = 0; s < Cfg::kStages; ++s)
          if ((armed >> s) & 1u) mbar_wait_drain(&sm.full[s], (armed_par >> s) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc0 = idesc_f16(kBM, 16, kBf16) & ~(0x3Fu << 17);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      int units = a.n_sh ? units_sh : 0;
      bool waited = false;
      for (int u = blockIdx.x; ok && advance(u, units, waited); u += gridDim.x) {
        const int tile = u / a.ksplit, sp = u % a.ksplit;
        const int kb0 = sp * KB / a.ksplit, kb1 = (sp + 1) * KB / a.ksplit;
        const TileEntry te = entry_of(tile / mblocks);
        const uint32_t idesc = idesc0 | (static_cast<uint32_t>(round16(te.nrows) >> 3) << 17);
        if (!mbar_wait(&sm.tempty[acc], acc_phase ^ 1u, ab)) break;
        tc_fence_after_sync();
        const uint32_t d_g = tmem_base + acc * Cfg::kAccCols;
        const uint32_t d_u = d_g + BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&sm.full[stage], phase, ab)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t st = smem_u32(sm.tiles + stage * Cfg::kStageBytes);
          const uint64_t dg = sw128_kmajor_desc(st);
          const uint64_t du = sw128_kmajor_desc(st + kATileBytes);
          const uint64_t db = sw128_kmajor_desc(st + 2 * kATileBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint32_t accum = (kb > kb0 || k > 0) ? 1u : 0u;
            umma_f16(d_g, dg + 2 * k, db + 2 * k, idesc, accum);
            umma_f16(d_u, du + 2 * k, db + 2 * k, idesc, accum);
          }
          umma_commit(&sm.empty[stage]);
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&sm.tfull[acc]);
        if (Cfg::kAccStages == 2) {
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        } else {
          acc_phase ^= 1u;
        }
      }
      // every MMA issued has completed before TMEM is freed
      umma_commit(sm.drain);
      mbar_wait_drain(sm.drain, 0);
    }
  } else {
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    int units = a.n_sh ? units_sh : 0;
    bool waited = false;
    for (int u = blockIdx.x; advance(u, units, waited); u += gridDim.x) {
      const int tile = u / a.ksplit;
      const TileEntry te = entry_of(tile / mblocks);
      const int mb = tile % mblocks;
      if (a.ksplit > 1) {
        // Split along K: this unit's partial G and U go to global memory; the
        // last unit of the tile to finish adds the partials up in split order
        // (so the sum is the same whichever unit is last) and applies the
        // SwiGLU.  Nothing waits on another CTA: the counter only decides who
        // finishes.  Every epilogue warp reaches every epilogue_bar(), also
        // after a failed wait, so a timeout cannot strand one at a barrier.
        const bool ok_w = __all_sync(0xffffffffu, mbar_wait(&sm.tfull[acc], acc_phase, ab));
        if (!ok_w && lane == 0) sm.split_flags[0] = 1;
        epilogue_bar();
        if (sm.split_flags[0]) break;
        tc_fence_after_sync();
        const int fl = q * 32 + lane;
        const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * Cfg::kAccCols;
        const int n = round16(te.nrows);
        float* pu = a.partial + static_cast<size_t>(u) * 2 * BN * kBM;
        for (int c0 = 0; c0 < n; c0 += 16) {
          uint32_t g[16], uv[16];
          tmem_ld_32x32b_x16(tq + c0, g);
          tmem_ld_32x32b_x16(tq + BN + c0, uv);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            pu[static_cast<size_t>(c0 + i) * kBM + fl] = __uint_as_float(g[i]);
            pu[static_cast<size_t>(BN + c0 + i) * kBM + fl] = __uint_as_float(uv[i]);
          }
        }
        tc_fence_before_sync();
        mbar_arrive(&sm.tempty[acc]);
        __threadfence();
        epilogue_bar();
        if (threadIdx.x == kEpiThread0)
          sm.split_flags[1] = atomicAdd(&a.counters[tile], 1) == a.ksplit - 1;
        epilogue_bar();
        if (sm.split_flags[1]) {
          __threadfence();
          const int f = mb * kBM + fl;
          const float* pt = a.partial + static_cast<size_t>(tile) * a.ksplit * 2 * BN * kBM;
          if (f < a.I) {
            // 16 token columns at a time: 32 independent loads per split step
            for (int c0 = 0; c0 < te.nrows; c0 += 16) {
              float gs[16], us[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) gs[i] = us[i] = 0.f;
              for (int p2 = 0; p2 < a.ksplit; ++p2) {
                const float* pp = pt + static_cast<size_t>(p2) * 2 * BN * kBM;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  gs[i] += __ldcg(pp + static_cast<size_t>(c0 + i) * kBM + fl);
                  us[i] += __ldcg(pp + static_cast<size_t>(BN + c0 + i) * kBM + fl);
                }
              }
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int c = c0 + i;
                if (c >= te.nrows || te.row0 + c >= a.total_rows) break;
                const float hv = clamped_swiglu(gs[i], us[i]);
                const size_t o = static_cast<size_t>(te.row0 + c) * a.I + f;
                if (kBf16) {
                  const __nv_bfloat16 hi = __float2bfloat16_rn(hv);
                  const __nv_bfloat16 lo = __float2bfloat16_rn(hv - __bfloat162float(hi));
                  static_cast<__nv_bfloat16*>(a.h0)[o] = hi;
                  static_cast<__nv_bfloat16*>(a.h1)[o] = lo;
                } else {
                  static_cast<__half*>(a.h0)[o] = __float2half_rn(hv);
                }
              }
            }
          }
          if (threadIdx.x == kEpiThread0) a.counters[tile] = 0;
        }
        epilogue_bar();  // the flags are read before the next unit rewrites them
        if (Cfg::kAccStages == 2) {
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        } else {
          acc_phase ^= 1u;
        }
        continue;
      }
      // warp-uniform outcome: tcgen05.ld below is .sync.aligned
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.tfull[acc], acc_phase, ab))) break;
      tc_fence_after_sync();
      const int f = mb * kBM + q * 32 + lane;
      const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * Cfg::kAccCols;
      const int n = round16(te.nrows);
      for (int c0 = 0; c0 < n; c0 += 16) {
        uint32_t g[16], u[16];
        tmem_ld_32x32b_x16(tq + c0, g);
        tmem_ld_32x32b_x16(tq + BN + c0, u);
        tmem_ld_wait();
        if (f < a.I) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = c0 + i;
            if (c < te.nrows && te.row0 + c < a.total_rows) {
              const float hv = clamped_swiglu(__uint_as_float(g[i]), __uint_as_float(u[i]));
              const size_t o = static_cast<size_t>(te.row0 + c) * a.I + f;
              if (kBf16) {
                const __nv_bfloat16 hi = __float2bfloat16_rn(hv);
                const __nv_bfloat16 lo = __float2bfloat16_rn(hv - __bfloat162float(hi));
                static_cast<__nv_bfloat16*>(a.h0)[o] = hi;
                static_cast<__nv_bfloat16*>(a.h1)[o] = lo;
              } else {
                static_cast<__half*>(a.h0)[o] = __float2half_rn(hv);
              }
            }
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&sm.tempty[acc]);
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

// ======================================================================
// Single-A GEMM: D = W[e] x B^T with one or two B operands per k-step
// (two = the hi/lo planes of h, summed into one accumulator).  Epilogues:
//   scatter-add  out[gather[r]][f] += roww[r] * D     (down, fused layer)
//   store rows   out[r][f] = D                         (down, y_perm)
//   router       out[r][f] = D + bias[f]               (router logits)
// ======================================================================
template <int BN, int NB, bool kBf16, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    down_kernel(const __grid_constant__ CUtensorMap tm_a,
                const __grid_constant__ CUtensorMap tm_a_shared,
                const __grid_constant__ CUtensorMap tm_b0,
                const __grid_constant__ CUtensorMap tm_b1, const DownArgs a) {
  using Cfg = DownCfg<BN, NB>;
  extern __shared__ uint8_t smem_raw[];
  const SmemCarve sm = carve(smem_raw, Cfg::kStages, Cfg::kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    init_barriers(sm, Cfg::kStages);
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_a_shared);
    tma_prefetch_desc(&tm_b0);
    if (NB == 2) tma_prefetch_desc(&tm_b1);
  }
  if (warp == 1) {
    tmem_alloc(sm.tmem_holder, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *sm.tmem_holder;
  const AbortState ab{sm.abort_flag, a.status, a.budget_ns};

  pdl_wait();
  pdl_launch_dependents();
  const int total = n_entries_of(a.table, a.dense_rows, BN) * a.mblocks;
  const int units = total * a.ksplit;  // ksplit > 1 only with the scatter-add epilogue
  const int KB = a.K / kBK;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        const int tile = u / a.ksplit, sp = u % a.ksplit;
        const int kb0 = sp * KB / a.ksplit, kb1 = (sp + 1) * KB / a.ksplit;
        const TileEntry te = entry_at(a.table, a.dense_rows, BN, tile / a.mblocks);
        const int mb = tile % a.mblocks;
        const bool sh = te.group == a.E;
        const CUtensorMap* ma = sh ? &tm_a_shared : &tm_a;
        const int ge = sh ? 0 : te.group;
        const int nchunks = (te.nrows + kChunkRows - 1) / kChunkRows;
        const uint32_t bytes = a.a_rows * kRowBytes + NB * nchunks * kChunkBytes;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&sm.empty[stage], phase ^ 1u, ab)) {
            ok = false;
            break;
          }
          uint8_t* st = sm.tiles + stage * Cfg::kStageBytes;
          mbar_arrive_expect_tx(&sm.full[stage], bytes);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          tma_load_3d(st, ma, &sm.full[stage], kb * kBK, mb * kBM, ge, pol_w);
          for (int c = 0; c < nchunks; ++c) {
            tma_load_2d(st + kATileBytes + c * kChunkBytes, &tm_b0, &sm.full[stage], kb * kBK,
                        te.row0 + c * kChunkRows, pol_x);
            if (NB == 2)
              tma_load_2d(st + kATileBytes + Cfg::kBTileBytes + c * kChunkBytes, &tm_b1,
                          &sm.full[stage], kb * kBK, te.row0 + c * kChunkRows, pol_x);
          }
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < Cfg::kStages; ++s)
        if ((armed >> s) & 1u) mbar_wait_drain(&sm.full[s], (armed_par >> s) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc0 = idesc_f16(kBM, 16, kBf16) & ~(0x3Fu << 17);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        const int tile = u / a.ksplit, sp = u % a.ksplit;
        const int kb0 = sp * KB / a.ksplit, kb1 = (sp + 1) * KB / a.ksplit;
        const TileEntry te = entry_at(a.table, a.dense_rows, BN, tile / a.mblocks);
        const uint32_t idesc = idesc0 | (static_cast<uint32_t>(round16(te.nrows) >> 3) << 17);
        if (!mbar_wait(&sm.tempty[acc], acc_phase ^ 1u, ab)) break;
        tc_fence_after_sync();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&sm.full[stage], phase, ab)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t st = smem_u32(sm.tiles + stage * Cfg::kStageBytes);
          const uint64_t da = sw128_kmajor_desc(st);
          const uint64_t db0 = sw128_kmajor_desc(st + kATileBytes);
          const uint64_t db1 = sw128_kmajor_desc(st + kATileBytes + Cfg::kBTileBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            umma_f16(d, da + 2 * k, db0 + 2 * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
            if (NB == 2) umma_f16(d, da + 2 * k, db1 + 2 * k, idesc, 1u);
          }
          umma_commit(&sm.empty[stage]);
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&sm.tfull[acc]);
        if (Cfg::kAccStages == 2) {
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        } else {
          acc_phase ^= 1u;
        }
      }
      umma_commit(sm.drain);
      mbar_wait_drain(sm.drain, 0);
    }
  } else {
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const int tile = u / a.ksplit;
      const TileEntry te = entry_at(a.table, a.dense_rows, BN, tile / a.mblocks);
      const int mb = tile % a.mblocks;
      // warp-uniform outcome: tcgen05.ld below is .sync.aligned
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.tfull[acc], acc_phase, ab))) break;
      tc_fence_after_sync();
      const int f = mb * kBM + q * 32 + lane;
      const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      const int n = round16(te.nrows);
      const float fbias = (EPI == kEpiRouter && f < a.N_out) ? a.bias[f] : 0.f;
      for (int c0 = 0; c0 < n; c0 += 16) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(tq + c0, v);
        tmem_ld_wait();
        if (f < a.N_out) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = c0 + i;
            const int r = te.row0 + c;
            if (c < te.nrows && r < a.total_rows) {
              const float d = __uint_as_float(v[i]);
              if (EPI == kEpiScatterAdd) {
                const int t = a.gather[r];
                if (t >= 0 && t < a.out_rows)
                  atomicAdd(a.out + static_cast<size_t>(t) * a.N_out + f, a.roww[r] * d);
              } else if (EPI == kEpiStoreRows) {
                a.out[static_cast<size_t>(r) * a.N_out + f] = d;
              } else {
                a.out[static_cast<size_t>(r) * a.N_out + f] = d + fbias;
              }
            }
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&sm.tempty[acc]);
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

// ======================================================================
// The decode FFN in one persistent launch (bf16 weights, scatter-add
// output): the gate/up units and the down units of a layer call in one unit
// list, handed out in list order from a counter in global memory (a CTA
// takes its next unit when it starts the current one):
//   [gate/up, shared expert]                            needs no routing
//   [gate/up, routed] [down, shared expert] [down, routed]   after the routing wait
// A down unit of entry i reads the h rows that the gate/up units of entry i
// write.  In place of a kernel boundary, the epilogue of each finished
// gate/up tile raises the entry's counter (after its h stores, release) and
// the producer of a down unit waits for the counter to count every gate/up
// tile of the entry (acquire) before it loads h.  Every dependency points to
// an earlier unit of the list, handed out before it to a CTA that runs its
// units in the order it took them, so the waits end once every CTA of the
// launch is resident (grid <= SMs, one CTA per SM); they are bounded like
// the mbarrier waits.  Handing units out (rather than a fixed stride) keeps
// the CTAs' byte counts within one unit of each other (measured: 4 or 5 of
// the 2 MB gate/up units per CTA at 8 tokens with a fixed stride).  What this buys
// over two launches: a CTA goes on from its last gate/up unit to its first
// down unit at once, where the second launch waited for the slowest gate/up
// CTA to finish and then filled its pipelines from nothing.  (Down units of
// the shared expert placed before the routing wait stalled their CTAs until
// the shared gate/up was done and left them behind the others: measured.)
// The last CTA to finish clears the counters for the next call.
// ======================================================================
// A down unit covers two 128-row blocks of the output features (256 rows of
// the down weights) against one h tile, so that a down stage carries as many
// weight bytes as a gate/up stage (two 16 KB tiles) and each h tile serves
// twice the weights.
template <int BN>
struct FfnCfg {
  static constexpr int kGuBytes = 2 * kATileBytes + BN * kRowBytes;      // A gate, A up, x rows
  static constexpr int kDnBytes = 2 * kATileBytes + 2 * BN * kRowBytes;  // 2 A down, h hi, h lo
  static constexpr int kStageBytes = kGuBytes > kDnBytes ? kGuBytes : kDnBytes;
  static constexpr int kStages = cmin(8, kStageBudget / kStageBytes);
  static constexpr int kAccCols = 2 * BN;  // gate/up: G then U; down: both row blocks
  static constexpr int kAccStages = (4 * BN <= 512) ? 2 : 1;
  static constexpr int kTmemCols = ceil_pow2_32(kAccStages * kAccCols);
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256;
  static_assert(kStageBytes % 1024 == 0 && (BN * kRowBytes) % 1024 == 0,
                "stage tiles must stay 1024-byte aligned");
};

constexpr int kDnRows = 2 * kBM;  // output features per down unit

struct FfnArgs {
  const int32_t* table;  // routed entries first, the shared group's entries last
  const int32_t* xrows;  // gate/up token rows gathered from x (null: x_perm boxes)
  int H, I, E, total_rows, T;
  int n_sh, sh_row0;     // shared entries (rows sh_row0 + t, token rows x[t])
  int ks_g, ks_d;        // units per tile along K: gate/up (over H), down (over I)
  float* partial;        // ks_g > 1: fp32 partial G/U per gate/up unit
  int* counters;         // ks_g > 1: finished units per gate/up tile
  int* ready;            // [n_ready]: finished gate/up tiles per entry, then [n_ready]:
  int n_ready;           // finished CTAs; all zero between calls
  int* work;             // next unit of the list to hand out (ready + n_ready + 1)
  void* h0;
  void* h1;
  const int32_t* gather;
  const float* roww;
  float* out;
  int out_rows;
  int* status;
  uint64_t budget_ns;
};

constexpr int kUnitRing = 16;  // units the producer may run ahead of the epilogue

struct UnitQueue {
  int slot;
  uint32_t phase;
  __device__ __forceinline__ void next() {
    if (++slot == kUnitRing) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

struct FfnUnit {
  bool down;
  int ei;        // entry: the shared entries, then the table's routed entries
  TileEntry te;
  int mb, kb0, kb1;  // mb: 128-row block (gate/up) or pair of blocks (down)
  int gu;        // gate/up: ordinal among the gate/up units (its partial slot)
};

// Unit u of the list; nr = the routed entries (known after the routing wait,
// needed only past the shared gate/up units).
__device__ __forceinline__ FfnUnit ffn_unit(const FfnArgs& a, int BN, int u, int nr) {
  const int mbg = a.I / kBM, mbd = a.H / kDnRows, kbg = a.H / kBK, kbd = a.I / kBK;
  const int gs = a.n_sh * mbg * a.ks_g, gr = nr * mbg * a.ks_g;
  const int ds = a.n_sh * mbd * a.ks_d;
  FfnUnit f;
  int v;
  bool routed;
  if (u < gs) {
    f.down = false, routed = false, v = u;
  } else if (u < gs + gr) {
    f.down = false, routed = true, v = u - gs;
  } else if (u < gs + gr + ds) {
    f.down = true, routed = false, v = u - gs - gr;
  } else {
    f.down = true, routed = true, v = u - gs - gr - ds;
  }
  const int ks = f.down ? a.ks_d : a.ks_g, mbs = f.down ? mbd : mbg, kbs = f.down ? kbd : kbg;
  const int tile = v / ks, sp = v % ks, ent = tile / mbs;
  f.mb = tile % mbs;
  f.kb0 = sp * kbs / ks;
  f.kb1 = (sp + 1) * kbs / ks;
  if (routed) {
    f.ei = a.n_sh + ent;
    f.te = table_entry(a.table, ent);
  } else {
    f.ei = ent;
    f.te = TileEntry{a.E, a.sh_row0 + ent * BN, min(BN, a.T - ent * BN), a.n_sh};
  }
  f.gu = f.down ? -1 : u;  // the gate/up units lead the list
  return f;
}

// Units a role may take: before the routing wait the shared expert's gate/up
// units; at the first unit past them the role waits for the preceding
// kernels and counts the routed entries.  Every role walks the same list.
struct FfnWalk {
  int units, nr;
  bool counted;
};

__device__ __forceinline__ bool ffn_more(const FfnArgs& a, int u, FfnWalk& w) {
  if (u < w.units) return true;
  if (w.counted) return false;
  pdl_wait();
  w.counted = true;
  w.nr = a.table[0] - a.n_sh;
  w.units += w.nr * (a.I / kBM) * a.ks_g + (w.nr + a.n_sh) * (a.H / kDnRows) * a.ks_d;
  return u < w.units;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    decode_ffn_kernel(const __grid_constant__ CUtensorMap tm_gate,
                      const __grid_constant__ CUtensorMap tm_up,
                      const __grid_constant__ CUtensorMap tm_sgate,
                      const __grid_constant__ CUtensorMap tm_sup,
                      const __grid_constant__ CUtensorMap tm_x,
                      const __grid_constant__ CUtensorMap tm_xs,
                      const __grid_constant__ CUtensorMap tm_down,
                      const __grid_constant__ CUtensorMap tm_sdown,
                      const __grid_constant__ CUtensorMap tm_h0,
                      const __grid_constant__ CUtensorMap tm_h1, const FfnArgs a) {
  using Cfg = FfnCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  // the unit queue: the producer publishes each unit it takes, the MMA and
  // epilogue roles follow in the same order; the epilogue frees the slot
  __shared__ int s_unit[kUnitRing];
  __shared__ uint64_t s_uf[kUnitRing], s_ue[kUnitRing];
  const SmemCarve sm = carve(smem_raw, Cfg::kStages, Cfg::kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(&s_uf[i], 1);
      mbar_init(&s_ue[i], 1);
    }
    init_barriers(sm, Cfg::kStages);
    tma_prefetch_desc(&tm_gate);
    tma_prefetch_desc(&tm_up);
    tma_prefetch_desc(&tm_sgate);
    tma_prefetch_desc(&tm_sup);
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_xs);
    tma_prefetch_desc(&tm_down);
    tma_prefetch_desc(&tm_sdown);
    tma_prefetch_desc(&tm_h0);
    tma_prefetch_desc(&tm_h1);
  }
  if (warp == 1) {
    tmem_alloc(sm.tmem_holder, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *sm.tmem_holder;
  const AbortState ab{sm.abort_flag, a.status, a.budget_ns};
  pdl_launch_dependents();
  const int mbg = a.I / kBM;
  const int pre_units = a.n_sh * mbg * a.ks_g;

  if (warp == 0) {
    // Producer.  Lane 0 arms the stages and loads the weight tiles, the x
    // rows in 16-row boxes (x for the shared entries, x_perm otherwise) and
    // the h rows of down units; with a.xrows the lanes gather the routed
    // entries' token rows straight from x (tile::gather4, rows 4L .. 4L+3).
    const bool gat = a.xrows != nullptr;
    if (gat || lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_par = 0;
      bool ok = true;
      FfnWalk wk{pre_units, 0, false};
      UnitQueue uq{0, 0};
      int u = lane == 0 ? atomicAdd(a.work, 1) : 0;
      if (gat) u = __shfl_sync(0xffffffffu, u, 0);
      while (ok) {
        const bool end = !ffn_more(a, u, wk);
        bool go = true;
        if (lane == 0) {
          go = mbar_wait(&s_ue[uq.slot], uq.phase ^ 1u, ab);
          if (go) {
            s_unit[uq.slot] = end ? -1 : u;
            mbar_arrive(&s_uf[uq.slot]);
          }
        }
        if (gat) go = __shfl_sync(0xffffffffu, go, 0);
        uq.next();
        if (!go || end) break;
        const FfnUnit f = ffn_unit(a, BN, u, wk.nr);
        const TileEntry& te = f.te;
        const bool sh = te.group == a.E;
        const int ge = sh ? 0 : te.group;
        const int nchunks = (te.nrows + kChunkRows - 1) / kChunkRows;
        if (f.down) {
          // h of the entry: every gate/up tile of it has stored its rows
          bool go = true;
          if (lane == 0) {
            go = wait_counter(&a.ready[f.ei], mbg, ab);
            if (go) fence_proxy_async_global();
          }
          if (gat) go = __shfl_sync(0xffffffffu, go, 0);
          if (!go) break;
          const CUtensorMap* ma = sh ? &tm_sdown : &tm_down;
          const uint32_t bytes = 2u * kATileBytes + 2u * nchunks * kChunkBytes;
          for (int kb = f.kb0; kb < f.kb1; ++kb) {
            uint8_t* st = sm.tiles + stage * Cfg::kStageBytes;
            go = true;
            if (lane == 0) {
              go = mbar_wait(&sm.empty[stage], phase ^ 1u, ab);
              if (go) {
                mbar_arrive_expect_tx(&sm.full[stage], bytes);
                armed |= 1u << stage;
                armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                tma_load_3d(st, ma, &sm.full[stage], kb * kBK, f.mb * kDnRows, ge, pol_w);
                tma_load_3d(st + kATileBytes, ma, &sm.full[stage], kb * kBK,
                            f.mb * kDnRows + kBM, ge, pol_w);
                for (int c = 0; c < nchunks; ++c) {
                  tma_load_2d(st + 2 * kATileBytes + c * kChunkBytes, &tm_h0, &sm.full[stage],
                              kb * kBK, te.row0 + c * kChunkRows, pol_x);
                  tma_load_2d(st + 2 * kATileBytes + BN * kRowBytes + c * kChunkBytes, &tm_h1,
                              &sm.full[stage], kb * kBK, te.row0 + c * kChunkRows, pol_x);
                }
              }
            }
            if (gat) go = __shfl_sync(0xffffffffu, go, 0);
            if (!go) {
              ok = false;
              break;
            }
            if (++stage == Cfg::kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          // the next unit, taken once this one's loads are issued (taking it
          // earlier let the first CTAs to start claim two units each while
          // the rest of the grid was still being scheduled: measured)
          u = lane == 0 ? atomicAdd(a.work, 1) : 0;
          if (gat) u = __shfl_sync(0xffffffffu, u, 0);
          continue;
        }
        const CUtensorMap* mg = sh ? &tm_sgate : &tm_gate;
        const CUtensorMap* mu = sh ? &tm_sup : &tm_up;
        const bool gat_u = gat && !sh;
        const int ngather = (te.nrows + 3) / 4;
        int tok[4] = {0, 0, 0, 0};
        if (gat_u && lane < ngather) {
#pragma unroll
          for (int j = 0; j < 4; ++j) tok[j] = a.xrows[te.row0 + min(4 * lane + j, te.nrows - 1)];
        }
        const uint32_t bytes = 2u * kATileBytes +
                               (gat_u ? ngather * 4 * kRowBytes : nchunks * kChunkBytes);
        const bool issuer = gat_u && lane < ngather;
        for (int kb = f.kb0; kb < f.kb1; ++kb) {
          uint8_t* st = sm.tiles + stage * Cfg::kStageBytes;
          bool go = true;
          if (lane == 0) {
            go = mbar_wait(&sm.empty[stage], phase ^ 1u, ab);
            if (go) {
              mbar_arrive_expect_tx(&sm.full[stage], bytes);
              armed |= 1u << stage;
              armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
              tma_load_3d(st, mg, &sm.full[stage], kb * kBK, f.mb * kBM, ge, pol_w);
              tma_load_3d(st + kATileBytes, mu, &sm.full[stage], kb * kBK, f.mb * kBM, ge, pol_w);
              if (sh)
                for (int c = 0; c < nchunks; ++c)
                  tma_load_2d(st + 2 * kATileBytes + c * kChunkBytes, &tm_xs, &sm.full[stage],
                              kb * kBK, te.row0 - a.sh_row0 + c * kChunkRows, pol_x);
              else if (!gat)
                for (int c = 0; c < nchunks; ++c)
                  tma_load_2d(st + 2 * kATileBytes + c * kChunkBytes, &tm_x, &sm.full[stage],
                              kb * kBK, te.row0 + c * kChunkRows, pol_x);
            }
          }
          if (gat) go = __shfl_sync(0xffffffffu, go, 0);
          if (!go) {
            ok = false;
            break;
          }
          if (issuer)
            tma_gather4_2d(st + 2 * kATileBytes + lane * 4 * kRowBytes, &tm_x, &sm.full[stage],
                           kb * kBK, tok[0], tok[1], tok[2], tok[3], pol_x);
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        u = lane == 0 ? atomicAdd(a.work, 1) : 0;
        if (gat) u = __shfl_sync(0xffffffffu, u, 0);
      }
      // every copy issued has landed before the CTA may exit
      if (lane == 0)
        for (int s = 0; s < Cfg::kStages; ++s)
          if ((armed >> s) & 1u) mbar_wait_drain(&sm.full[s], (armed_par >> s) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc0 = idesc_f16(kBM, 16, true) & ~(0x3Fu << 17);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      FfnWalk wk{pre_units, 0, false};
      UnitQueue uq{0, 0};
      while (ok) {
        if (!mbar_wait(&s_uf[uq.slot], uq.phase, ab)) break;
        const int u = s_unit[uq.slot];
        uq.next();
        if (u < 0) break;
        ffn_more(a, u, wk);  // past the shared units: the routing wait, the routed count
        const FfnUnit f = ffn_unit(a, BN, u, wk.nr);
        const uint32_t idesc = idesc0 | (static_cast<uint32_t>(round16(f.te.nrows) >> 3) << 17);
        if (!mbar_wait(&sm.tempty[acc], acc_phase ^ 1u, ab)) break;
        tc_fence_after_sync();
        const uint32_t d0 = tmem_base + acc * Cfg::kAccCols;
        for (int kb = f.kb0; kb < f.kb1; ++kb) {
          if (!mbar_wait(&sm.full[stage], phase, ab)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t st = smem_u32(sm.tiles + stage * Cfg::kStageBytes);
          const uint32_t first = kb > f.kb0 ? 1u : 0u;
          if (f.down) {
            const uint64_t da0 = sw128_kmajor_desc(st);
            const uint64_t da1 = sw128_kmajor_desc(st + kATileBytes);
            const uint64_t db0 = sw128_kmajor_desc(st + 2 * kATileBytes);
            const uint64_t db1 = sw128_kmajor_desc(st + 2 * kATileBytes + BN * kRowBytes);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              const uint32_t accum = (first || k > 0) ? 1u : 0u;
              umma_f16(d0, da0 + 2 * k, db0 + 2 * k, idesc, accum);
              umma_f16(d0, da0 + 2 * k, db1 + 2 * k, idesc, 1u);
              umma_f16(d0 + BN, da1 + 2 * k, db0 + 2 * k, idesc, accum);
              umma_f16(d0 + BN, da1 + 2 * k, db1 + 2 * k, idesc, 1u);
            }
          } else {
            const uint64_t dg = sw128_kmajor_desc(st);
            const uint64_t du = sw128_kmajor_desc(st + kATileBytes);
            const uint64_t db = sw128_kmajor_desc(st + 2 * kATileBytes);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              const uint32_t accum = (first || k > 0) ? 1u : 0u;
              umma_f16(d0, dg + 2 * k, db + 2 * k, idesc, accum);
              umma_f16(d0 + BN, du + 2 * k, db + 2 * k, idesc, accum);
            }
          }
          umma_commit(&sm.empty[stage]);
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&sm.tfull[acc]);
        if (Cfg::kAccStages == 2) {
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        } else {
          acc_phase ^= 1u;
        }
      }
      // every MMA issued has completed before TMEM is freed
      umma_commit(sm.drain);
      mbar_wait_drain(sm.drain, 0);
    }
  } else {
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int fl = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    FfnWalk wk{pre_units, 0, false};
    UnitQueue uq{0, 0};
    for (;;) {
      const bool ok_u = __all_sync(0xffffffffu, mbar_wait(&s_uf[uq.slot], uq.phase, ab));
      if (!ok_u && lane == 0) sm.split_flags[0] = 1;
      epilogue_bar();
      if (sm.split_flags[0]) break;
      const int u = s_unit[uq.slot];
      const int slot = uq.slot;
      uq.next();
      if (u < 0) break;
      ffn_more(a, u, wk);
      const FfnUnit f = ffn_unit(a, BN, u, wk.nr);
      const TileEntry& te = f.te;
      // warp-uniform outcome: tcgen05.ld below is .sync.aligned; every
      // epilogue warp reaches every epilogue_bar(), also after a failed wait
      const bool ok_w = __all_sync(0xffffffffu, mbar_wait(&sm.tfull[acc], acc_phase, ab));
      if (!ok_w && lane == 0) sm.split_flags[0] = 1;
      epilogue_bar();
      if (sm.split_flags[0]) break;
      tc_fence_after_sync();
      const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * Cfg::kAccCols;
      const int n = round16(te.nrows);
      if (f.down) {
        // (past the routing wait: out is cleared, gather / roww are written)
        const int fo = f.mb * kDnRows + fl;
        for (int c0 = 0; c0 < n; c0 += 16) {
          uint32_t v0[16], v1[16];
          tmem_ld_32x32b_x16(tq + c0, v0);
          tmem_ld_32x32b_x16(tq + BN + c0, v1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = c0 + i;
            const int r = te.row0 + c;
            if (c < te.nrows && r < a.total_rows) {
              const int t = a.gather[r];
              if (t >= 0 && t < a.out_rows) {
                float* o = a.out + static_cast<size_t>(t) * a.H + fo;
                const float wr = a.roww[r];
                atomicAdd(o, wr * __uint_as_float(v0[i]));
                atomicAdd(o + kBM, wr * __uint_as_float(v1[i]));
              }
            }
          }
        }
        tc_fence_before_sync();
        mbar_arrive(&sm.tempty[acc]);
      } else {
        const int f_out = f.mb * kBM + fl;
        bool wrote = true;  // this unit stored its tile's h rows
        auto store_h = [&](int c, float g, float uu) {
          const float hv = clamped_swiglu(g, uu);
          const size_t o = static_cast<size_t>(te.row0 + c) * a.I + f_out;
          const __nv_bfloat16 hi = __float2bfloat16_rn(hv);
          const __nv_bfloat16 lo = __float2bfloat16_rn(hv - __bfloat162float(hi));
          static_cast<__nv_bfloat16*>(a.h0)[o] = hi;
          static_cast<__nv_bfloat16*>(a.h1)[o] = lo;
        };
        if (a.ks_g > 1) {
          // Split along K: the partial G and U go to global memory; the last
          // unit of the tile to finish adds the partials in split order and
          // applies the SwiGLU (nothing waits: the counter picks who finishes).
          const int tile = f.gu / a.ks_g;
          float* pu = a.partial + static_cast<size_t>(f.gu) * 2 * BN * kBM;
          for (int c0 = 0; c0 < n; c0 += 16) {
            uint32_t g[16], uv[16];
            tmem_ld_32x32b_x16(tq + c0, g);
            tmem_ld_32x32b_x16(tq + BN + c0, uv);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              pu[static_cast<size_t>(c0 + i) * kBM + fl] = __uint_as_float(g[i]);
              pu[static_cast<size_t>(BN + c0 + i) * kBM + fl] = __uint_as_float(uv[i]);
            }
          }
          tc_fence_before_sync();
          mbar_arrive(&sm.tempty[acc]);
          // the partials of all four warps are ordered before the count by
          // the barrier and the counting thread's release; its acquire
          // orders the finisher's partial loads after the other parts' counts
          epilogue_bar();
          if (threadIdx.x == kEpiThread0)
            sm.split_flags[1] = atom_acq_rel_gpu_add(&a.counters[tile], 1) == a.ks_g - 1;
          epilogue_bar();
          wrote = sm.split_flags[1] != 0;
          if (wrote) {
            const float* pt = a.partial + static_cast<size_t>(tile) * a.ks_g * 2 * BN * kBM;
            if (f_out < a.I) {
              for (int c0 = 0; c0 < te.nrows; c0 += 16) {
                float gs[16], us[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) gs[i] = us[i] = 0.f;
                for (int p2 = 0; p2 < a.ks_g; ++p2) {
                  const float* pp = pt + static_cast<size_t>(p2) * 2 * BN * kBM;
#pragma unroll
                  for (int i = 0; i < 16; ++i) {
                    gs[i] += __ldcg(pp + static_cast<size_t>(c0 + i) * kBM + fl);
                    us[i] += __ldcg(pp + static_cast<size_t>(BN + c0 + i) * kBM + fl);
                  }
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const int c = c0 + i;
                  if (c >= te.nrows || te.row0 + c >= a.total_rows) break;
                  store_h(c, gs[i], us[i]);
                }
              }
            }
            if (threadIdx.x == kEpiThread0) a.counters[tile] = 0;
          }
        } else {
          for (int c0 = 0; c0 < n; c0 += 16) {
            uint32_t g[16], uv[16];
            tmem_ld_32x32b_x16(tq + c0, g);
            tmem_ld_32x32b_x16(tq + BN + c0, uv);
            tmem_ld_wait();
            if (f_out < a.I) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int c = c0 + i;
                if (c < te.nrows && te.row0 + c < a.total_rows)
                  store_h(c, __uint_as_float(g[i]), __uint_as_float(uv[i]));
              }
            }
          }
          tc_fence_before_sync();
          mbar_arrive(&sm.tempty[acc]);
        }
        if (wrote) {
          // the tile's h rows (all four warps', ordered by the barrier) are
          // visible GPU-wide before the entry counts it
          epilogue_bar();
          if (threadIdx.x == kEpiThread0) {
            fence_proxy_async_global();
            red_release_gpu_add(&a.ready[f.ei], 1);
          }
        }
      }
      epilogue_bar();  // shared flags are read before the next unit rewrites them
      if (threadIdx.x == kEpiThread0) mbar_arrive(&s_ue[slot]);
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
  if (threadIdx.x == 0) {
    // the last CTA to finish clears the counters: every other CTA is past
    // all its waits and signals
    __threadfence();
    if (atomicAdd(&a.ready[a.n_ready], 1) == static_cast<int>(gridDim.x) - 1) {
      for (int i = 0; i < a.n_ready; ++i) a.ready[i] = 0;
      a.ready[a.n_ready] = 0;
      *a.work = 0;
      __threadfence();
    }
  }
}

__global__ void wait_selftest_kernel(int* status, uint64_t budget_ns) {
  __shared__ uint64_t bar;
  __shared__ int flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const AbortState ab{&flag, status, budget_ns};
    mbar_wait(&bar, 0, ab);  // nothing arrives: runs out of budget
  }
}

template <int BN, bool kBf16>
cudaError_t gateup_dispatch(const GateUpLaunch& L, cudaStream_t s) {
  using Cfg = GateUpCfg<BN>;
  auto kern = gateup_kernel<BN, kBf16>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (err != cudaSuccess) return err;
  GateUpArgs a{L.table,      L.xrows,  L.K,  L.I,          L.E,
               L.a_rows,     L.total_rows, L.n_sh, L.T, L.sh_row0,
               L.ksplit > 0 ? L.ksplit : 1, L.partial, L.counters, L.h0, L.h1, L.status,
               L.budget_ns};
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
  return cudaLaunchKernelEx(&cfg, kern, L.tm_gate, L.tm_up, L.tm_sgate, L.tm_sup, L.tm_x,
                            L.tm_xs, a);
}

template <int BN, int NB, bool kBf16, int EPI>
cudaError_t down_dispatch(const DownLaunch& L, cudaStream_t s) {
  using Cfg = DownCfg<BN, NB>;
  auto kern = down_kernel<BN, NB, kBf16, EPI>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (err != cudaSuccess) return err;
  DownArgs a{L.table, L.dense_rows, EPI == kEpiScatterAdd && L.ksplit > 1 ? L.ksplit : 1, L.K,
             L.N_out, L.mblocks, L.E, L.a_rows, L.total_rows, L.out_rows, L.gather, L.roww,
             L.bias, L.out, L.status, L.budget_ns};
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
  return cudaLaunchKernelEx(&cfg, kern, L.tm_a, L.tm_a_shared, L.tm_b0, L.tm_b1, a);
}

template <int BN>
cudaError_t ffn_dispatch(const FfnLaunch& L, cudaStream_t s) {
  using Cfg = FfnCfg<BN>;
  auto kern = decode_ffn_kernel<BN>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (err != cudaSuccess) return err;
  const GateUpLaunch& G = L.g;
  FfnArgs a{G.table,  G.xrows,    G.K,       G.I,         G.E,     G.total_rows, G.T,
            G.n_sh,   G.sh_row0,  G.ksplit > 0 ? G.ksplit : 1, L.ks_d > 0 ? L.ks_d : 1,
            G.partial, G.counters, L.ready,  L.n_ready,   L.ready + L.n_ready + 1,
            G.h0,     G.h1,       L.gather,
            L.roww,   L.out,      L.out_rows, G.status,   G.budget_ns};
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
  return cudaLaunchKernelEx(&cfg, kern, G.tm_gate, G.tm_up, G.tm_sgate, G.tm_sup, G.tm_x, G.tm_xs,
                            L.tm_down, L.tm_sdown, L.tm_h0, L.tm_h1, a);
}

template <int NB, bool kBf16, int EPI>
cudaError_t down_by_bn(const DownLaunch& L, cudaStream_t s) {
  switch (L.BN) {
    case 16: return down_dispatch<16, NB, kBf16, EPI>(L, s);
    case 32: return down_dispatch<32, NB, kBf16, EPI>(L, s);
    case 64: return down_dispatch<64, NB, kBf16, EPI>(L, s);
    case 128: return down_dispatch<128, NB, kBf16, EPI>(L, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_gateup(const GateUpLaunch& L, cudaStream_t s) {
  if (L.bf16) {
    switch (L.BN) {
      case 16: return gateup_dispatch<16, true>(L, s);
      case 32: return gateup_dispatch<32, true>(L, s);
      case 64: return gateup_dispatch<64, true>(L, s);
      case 128: return gateup_dispatch<128, true>(L, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (L.BN) {
    case 16: return gateup_dispatch<16, false>(L, s);
    case 32: return gateup_dispatch<32, false>(L, s);
    case 64: return gateup_dispatch<64, false>(L, s);
    case 128: return gateup_dispatch<128, false>(L, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_down(const DownLaunch& L, cudaStream_t s) {
  if (L.epilogue == kEpiRouter) {
    if (!L.bf16 || L.nb != 1) return cudaErrorInvalidValue;
    return down_by_bn<1, true, kEpiRouter>(L, s);
  }
  if (L.bf16) {
    if (L.nb != 2) return cudaErrorInvalidValue;
    return L.epilogue == kEpiScatterAdd ? down_by_bn<2, true, kEpiScatterAdd>(L, s)
                                        : down_by_bn<2, true, kEpiStoreRows>(L, s);
  }
  if (L.nb != 1) return cudaErrorInvalidValue;
  return L.epilogue == kEpiScatterAdd ? down_by_bn<1, false, kEpiScatterAdd>(L, s)
                                      : down_by_bn<1, false, kEpiStoreRows>(L, s);
}

cudaError_t launch_decode_ffn(const FfnLaunch& L, cudaStream_t s) {
  const GateUpLaunch& G = L.g;
  if (!G.bf16 || G.n_sh <= 0 || G.I % kBM != 0 || G.K % kDnRows != 0 || !L.ready || L.grid <= 0)
    return cudaErrorInvalidValue;
  switch (G.BN) {
    case 16: return ffn_dispatch<16>(L, s);
    case 32: return ffn_dispatch<32>(L, s);
    case 64: return ffn_dispatch<64>(L, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_wait_selftest(int* status, uint64_t budget_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, budget_ns);
  return cudaGetLastError();
}

}  // namespace moe
