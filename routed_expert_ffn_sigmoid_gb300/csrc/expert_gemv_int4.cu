// Grouped Int4 expert GEMVs on CUDA cores for decode-size tile entries (at
// most kGemvMaxRows token rows each): gate/up with the clamped SwiGLU, then
// down with the routing weight and the scatter-add into out (or the
// unweighted row store of the deterministic mode).
//
// Weights use the grouped fmt=4 Int4 format decoded as offset-binary,
// value = (nibble - 8) * scale, one bf16 scale per 32 reduction elements
// ("feat(glm53): add device-resident HIP backend for MI350P", section "Key
// changes"); the expert FFN follows "Add GLM-5.3-Flash (glm5next) support
// with ROCmFP mix qtypes (105/106)", section "MoE FFN (REAL routed expert
// execution)".
//
// Why CUDA cores.  An entry of one to eight token rows uses each weight only
// that many times, so the layer is a stream of weight bytes.  A tensor-core
// MMA needs every 4-bit code turned into an operand element first, and that
// conversion, not HBM, bounds the 8-bit tcgen05 kernels at these sizes.
// Here the codes enter 8-bit integer dot products (dp4a) as they are, after
// two masks per word of eight codes:
//   sum_{k in g} (n_k - 8) s_g a_k = s_g sigma_g (sum_k n_k q_k - 8 sum_k q_k)
// with q_k = round(a_k / sigma_g) a 16-bit integer under a power-of-two scale
// sigma_g per activation row and group g of 32 (the group's largest |a| lies
// in [2^14, 2^15) sigma_g), stored as a signed high byte and an unsigned low
// byte, q = 256 hi + lo.  Every group sum is an exact integer below 2^23 in
// magnitude, converted to fp32 once and scaled by s_g sigma_g; only the fp32
// sum over groups rounds.  A bf16 activation is exact in q when it lies
// within 2^-7 of its group's largest |a| (same exponent or up to seven
// below); smaller ones, and h (fp32), are off by at most half a quantum,
// 2^-15 of the group's largest |a| (2^-14 where q clamps to 32767).  Groups
// whose largest |a| is below 2^-100 count as zero.
//
// Activation planes, per row and group c of 32 elements: 64 bytes as four
// 16-byte words, [hi 0..15][hi 16..31][lo 0..15][lo 16..31] in the element
// order the code masks produce: within every aligned group of 8 elements,
// (0, 2, 4, 6) then (1, 3, 5, 7).  In shared memory, and for h in the
// workspace, the four words lie in four planes [row][word][c] so that lanes
// reading consecutive groups read consecutive 16-byte words.
//
// CTA = 8 warps, persistent over the units of the flat tile list (unit
// blockIdx.x, then every gridDim.x-th: the units of an entry, whose work
// grows with its rows, spread over many CTAs):
//   gate/up: unit = (entry, 32 features), one h scale group; a warp takes 4
//            features, one per pass (its gate and up rows), its lanes split
//            K = H in 16-byte code words (lane l: groups l, l + 32, ...);
//            after the SwiGLU the warp of token row t quantises the group
//            of 32 h values of row t.
//   down:    unit = (entry, 128 rows of H); each half-warp takes 4 rows (2
//            for 5..8 token rows or I > 1536) per pass, its lanes split
//            K = I (lane l: groups l, l + 16, ...).
// Lane partial sums are combined by a reduce-scatter across the lanes (one
// value per lane at the end), so that the epilogue runs on many lanes.
#include <cuda_bf16.h>
#include <stdint.h>

#include "gemm_common.cuh"
#include "moe_kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = kGemvMaxRows;                  // token rows per entry
constexpr int kUnitFeatures = 32;                    // gate/up features per unit
constexpr int kWarpFeatures = kUnitFeatures / kWarps;  // 4
constexpr int kDownWarpRows = 16;
constexpr int kDownUnitRows = kWarps * kDownWarpRows;  // 128

struct GemvArgs {
  const int32_t* table;
  int E, K, N_out, total_rows, out_rows;
  // gate/up: token rows of x (row r of an entry is x[xrows[r]]), bf16 [.][K]
  const uint16_t* x;
  const int32_t* xrows;
  // codes [E][N_out][K/2] and bf16 scales [E][N_out][K/32]: gate, up (or down
  // in slot 0); s*: the shared expert's
  const uint8_t* codes0;
  const uint8_t* codes1;
  const uint16_t* scale0;
  const uint16_t* scale1;
  const uint8_t* scodes0;
  const uint8_t* scodes1;
  const uint16_t* sscale0;
  const uint16_t* sscale1;
  // h planes [rows][4][I/32] x 16 B, sigma [rows][I/32], 8 sum q [rows][I/32]
  uint8_t* hq;
  float* hs;
  int32_t* hc;
  // down
  const int32_t* gather;
  const float* roww;
  float* out;
};

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// sum over one group of 32 weights (code words cw) of (n - 8) q, with the
// activation's planes av = [hi 0..3][hi 4..7][lo 0..3][lo 4..7] (words) and
// corr = 8 sum q.  Even codes come out of the mask 0x0F0F0F0F, odd codes of
// 0xF0F0F0F0 as 16 n: those sums are divided by 16 exactly at the end.
__device__ __forceinline__ int group_dot(const uint4& cw, const uint4 (&av)[4], int corr) {
  const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
  const uint32_t ah[8] = {av[0].x, av[0].y, av[0].z, av[0].w, av[1].x, av[1].y, av[1].z, av[1].w};
  const uint32_t al[8] = {av[2].x, av[2].y, av[2].z, av[2].w, av[3].x, av[3].y, av[3].z, av[3].w};
  int he = 0, ho = 0;
  uint32_t le = 0, lo = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t e = w[k] & 0x0F0F0F0Fu, o = w[k] & 0xF0F0F0F0u;
    he = dp4a_us(e, ah[2 * k], he);
    ho = dp4a_us(o, ah[2 * k + 1], ho);
    le = dp4a_uu(e, al[2 * k], le);
    lo = dp4a_uu(o, al[2 * k + 1], lo);
  }
  // |he| <= 16 * 15 * 128, |ho| <= 16 * 240 * 128, le, lo < 16 * 240 * 256:
  // no overflow; ho * 256 + lo is a multiple of 16
  const int even = he * 256 + static_cast<int>(le);
  const int odd16 = ho * 256 + static_cast<int>(lo);
  return even + (odd16 >> 4) - corr;
}

// The 16-bit quantisation of one group: inv = 1 / sigma, sigma (0 for a
// group that counts as zero).
struct GroupScale {
  float inv, sigma;
};

__device__ __forceinline__ GroupScale group_scale(float amax) {
  const uint32_t ef = __float_as_uint(amax) >> 23;  // biased exponent of the largest |a|
  if (ef < 27u) return GroupScale{0.f, 0.f};
  // amax in [2^e, 2^(e+1)), e = ef - 127: sigma = 2^(e - 14)
  return GroupScale{__uint_as_float((268u - ef) << 23), __uint_as_float((ef - 14u) << 23)};
}

__device__ __forceinline__ int quantise(float a, float inv) {
  const int q = __float2int_rn(a * inv);
  return max(-32767, min(32767, q));
}

// Position of element j (0..31) of a group in the plane words: word index
// (0..7) and byte within it.
__device__ __forceinline__ int plane_word(int j) { return 2 * (j >> 3) + (j & 1); }
__device__ __forceinline__ int plane_byte(int j) { return (j & 7) >> 1; }

// x rows of one entry -> activation planes in shared memory: one thread per
// (row, group).
__device__ __forceinline__ void stage_x_rows(const GemvArgs& a, const int* s_xrow, int nt,
                                             uint4* s_act, float* s_sig, int* s_corr) {
  const int nch = a.K / 32;
  for (int i = threadIdx.x; i < nt * nch; i += kThreads) {
    const int t = i / nch, c = i - t * nch;
    const uint4* src =
        reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(s_xrow[t]) * a.K + c * 32);
    uint32_t wv[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 v = __ldg(src + j);
      wv[4 * j] = v.x;
      wv[4 * j + 1] = v.y;
      wv[4 * j + 2] = v.z;
      wv[4 * j + 3] = v.w;
    }
    float av[32];
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      av[2 * j] = bf16_bits_to_float(wv[j] & 0xFFFFu);
      av[2 * j + 1] = bf16_bits_to_float(wv[j] >> 16);
      amax = fmaxf(amax, fmaxf(fabsf(av[2 * j]), fabsf(av[2 * j + 1])));
    }
    const GroupScale gs = group_scale(amax);
    uint32_t hw[8], lw[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) hw[j] = lw[j] = 0u;
    int sum = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int q = quantise(av[j], gs.inv);
      sum += q;
      const int w = plane_word(j), sh = 8 * plane_byte(j);
      hw[w] |= (static_cast<uint32_t>(q >> 8) & 0xFFu) << sh;
      lw[w] |= (static_cast<uint32_t>(q) & 0xFFu) << sh;
    }
    uint4* dst = s_act + static_cast<size_t>(t) * 4 * nch + c;
    dst[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    dst[nch] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
    dst[2 * nch] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    dst[3 * nch] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
    s_sig[t * nch + c] = gs.sigma;
    s_corr[t * nch + c] = 8 * sum;
  }
}

// Sum of V values per lane over groups of G lanes (G = 32 or 16), scattered:
// afterwards lane l of a group holds value (l % G) / (G / V) summed over the
// group's lanes.
template <int V, int G>
__device__ __forceinline__ float reduce_scatter(float (&v)[V], int lane) {
  constexpr int kSteps = V >= 32 ? 5 : V >= 16 ? 4 : V >= 8 ? 3 : V >= 4 ? 2 : V >= 2 ? 1 : 0;
  static_assert((1 << kSteps) == V && V <= G, "V: a power of two up to G");
#pragma unroll
  for (int s = 0; s < kSteps; ++s) {
    const int w = G >> (s + 1);
    const int half = V >> (s + 1);
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  float r = v[0];
#pragma unroll
  for (int w = G >> (kSteps + 1); w >= 1; w >>= 1) r += __shfl_xor_sync(0xffffffffu, r, w);
  return r;
}

// ---------------------------------------------------------------- gate/up

// One pass of a warp over R weight rows (gate and up of R / 2 features f0..)
// for NT token rows (nt of them live); MC code words per lane and row.
template <int MC, int NT, int R>
__device__ __forceinline__ void gateup_pass(const GemvArgs& a, const uint8_t* cg,
                                            const uint8_t* cu, const uint16_t* sg,
                                            const uint16_t* su, int f0, int nt,
                                            const uint4* s_act, const float* s_sig,
                                            const int* s_corr, float* s_h, int fl0) {
  const int lane = threadIdx.x & 31;
  const int nch = a.K / 32;
  const size_t crow = a.K / 2;
  uint4 cw[R][MC];
  float sw[R][MC];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const size_t f = static_cast<size_t>(f0 + (r >> 1));
    const uint8_t* cb = ((r & 1) ? cu : cg) + f * crow;
    const uint16_t* sb = ((r & 1) ? su : sg) + f * nch;
#pragma unroll
    for (int m = 0; m < MC; ++m) {
      cw[r][m] = ld_stream16(cb + static_cast<size_t>(lane + 32 * m) * 16);
      sw[r][m] = bf16_bits_to_float(__ldg(sb + lane + 32 * m));
    }
  }
  float acc[R * NT];
#pragma unroll
  for (int i = 0; i < R * NT; ++i) acc[i] = 0.f;
#pragma unroll
  for (int m = 0; m < MC; ++m) {
    const int c = lane + 32 * m;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < nt) {
        const uint4* ap = s_act + static_cast<size_t>(t) * 4 * nch + c;
        const uint4 av[4] = {ap[0], ap[nch], ap[2 * nch], ap[3 * nch]};
        const float sig = s_sig[t * nch + c];
        const int corr = s_corr[t * nch + c];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int v = group_dot(cw[r][m], av, corr);
          acc[r * NT + t] = fmaf(static_cast<float>(v), sw[r][m] * sig, acc[r * NT + t]);
        }
      }
    }
  }
  constexpr int V = R * NT;
  const float val = reduce_scatter<V, 32>(acc, lane);
  // lane l holds value idx = l / (32 / V): row idx / NT, token row idx % NT;
  // the up row of the same feature sits 32 / R lanes further on
  const float up = __shfl_down_sync(0xffffffffu, val, 32 / R);
  constexpr int kLanesPerValue = 32 / V;
  const int idx = lane / kLanesPerValue;
  const int r = idx / NT, t = idx % NT;
  if (lane % kLanesPerValue == 0 && (r & 1) == 0 && t < nt)
    s_h[t * kUnitFeatures + fl0 + (r >> 1)] = clamped_swiglu(val, up);
}

template <int MC, int NT>
__device__ __forceinline__ void gateup_unit(const GemvArgs& a, const TileEntry& te, int fb, int nt,
                                            const uint4* s_act, const float* s_sig,
                                            const int* s_corr, float* s_h) {
  const int warp = threadIdx.x >> 5;
  const bool sh = te.group == a.E;
  const size_t e = sh ? 0 : static_cast<size_t>(te.group);
  const size_t cexp = static_cast<size_t>(a.N_out) * (a.K / 2);
  const size_t sexp = static_cast<size_t>(a.N_out) * (a.K / 32);
  const uint8_t* cg = (sh ? a.scodes0 : a.codes0) + e * cexp;
  const uint8_t* cu = (sh ? a.scodes1 : a.codes1) + e * cexp;
  const uint16_t* sg = (sh ? a.sscale0 : a.scale0) + e * sexp;
  const uint16_t* su = (sh ? a.sscale1 : a.scale1) + e * sexp;
  constexpr int R = 2;  // rows per pass: gate and up of one feature
#pragma unroll 1
  for (int p = 0; p < kWarpFeatures / (R / 2); ++p) {
    const int fl0 = warp * kWarpFeatures + p * (R / 2);  // feature within the unit
    gateup_pass<MC, NT, R>(a, cg, cu, sg, su, fb * kUnitFeatures + fl0, nt, s_act, s_sig, s_corr,
                           s_h, fl0);
  }
}

template <int MC>
__global__ void __launch_bounds__(kThreads, 2) int4_gemv_gateup_kernel(const GemvArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int nch = a.K / 32;
  uint4* s_act = reinterpret_cast<uint4*>(smem);
  float* s_sig = reinterpret_cast<float*>(s_act + static_cast<size_t>(kRows) * 4 * nch);
  int* s_corr = reinterpret_cast<int*>(s_sig + kRows * nch);
  float* s_h = reinterpret_cast<float*>(s_corr + kRows * nch);
  __shared__ int s_xrow[kRows];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_wait();
  pdl_launch_dependents();
  const int nfb = a.N_out / kUnitFeatures;
  const int total = a.table[0] * nfb;
  int staged = -1;  // entry whose rows s_act holds
  for (int u = blockIdx.x; u < total; u += gridDim.x) {
    const int ei = u / nfb, fb = u - ei * nfb;
    const TileEntry te = table_entry(a.table, ei);
    const int nt = min(te.nrows, kRows);
    if (ei != staged) {
      __syncthreads();  // every warp is done with the previous rows
      if (threadIdx.x < kRows) {
        const int r = te.row0 + threadIdx.x;
        const int tok = (threadIdx.x < nt && r < a.total_rows) ? a.xrows[r] : 0;
        s_xrow[threadIdx.x] = (tok >= 0 && tok < a.out_rows) ? tok : 0;
      }
      __syncthreads();
      stage_x_rows(a, s_xrow, nt, s_act, s_sig, s_corr);
      __syncthreads();
      staged = ei;
    }
    if (nt <= 1)
      gateup_unit<MC, 1>(a, te, fb, nt, s_act, s_sig, s_corr, s_h);
    else if (nt <= 2)
      gateup_unit<MC, 2>(a, te, fb, nt, s_act, s_sig, s_corr, s_h);
    else if (nt <= 4)
      gateup_unit<MC, 4>(a, te, fb, nt, s_act, s_sig, s_corr, s_h);
    else
      gateup_unit<MC, 8>(a, te, fb, nt, s_act, s_sig, s_corr, s_h);
    __syncthreads();  // s_h complete
    // the warp of token row t quantises row t's 32 h values (one group)
    if (warp < nt) {
      const int t = warp;
      const float hv = s_h[t * kUnitFeatures + lane];
      float amax = fabsf(hv);
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, w));
      const GroupScale gs = group_scale(amax);
      const int q = quantise(hv, gs.inv);
      int sum = q;
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, w);
      // lanes 0..15 assemble plane word (lane & 7) of the hi (lanes 0..7) or
      // lo (8..15) plane from the four lanes whose elements it holds
      const int wi = lane & 7, k = wi >> 1, par = wi & 1;
      const bool lo_plane = (lane & 8) != 0;
      uint32_t word = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int qs = __shfl_sync(0xffffffffu, q, 8 * k + 2 * b + par);
        const uint32_t byte = lo_plane ? (static_cast<uint32_t>(qs) & 0xFFu)
                                       : (static_cast<uint32_t>(qs >> 8) & 0xFFu);
        word |= byte << (8 * b);
      }
      const int rr = te.row0 + t;
      const int nchI = a.N_out / 32;
      if (rr < a.total_rows) {
        if (lane < 16) {
          const int plane = (lo_plane ? 2 : 0) + (wi >> 2);
          uint32_t* dst = reinterpret_cast<uint32_t*>(
              a.hq + (static_cast<size_t>(rr) * 4 * nchI + static_cast<size_t>(plane) * nchI + fb) * 16);
          dst[wi & 3] = word;
        }
        if (lane == 0) {
          a.hs[static_cast<size_t>(rr) * nchI + fb] = gs.sigma;
          a.hc[static_cast<size_t>(rr) * nchI + fb] = 8 * sum;
        }
      }
    }
    __syncthreads();  // s_h is read before the next unit writes it
  }
}

// ---------------------------------------------------------------- down

template <int MC, int NT, int EPI>
__device__ __forceinline__ void down_unit(const GemvArgs& a, const TileEntry& te, int jb, int nt,
                                          const uint4* s_act, const float* s_sig,
                                          const int* s_corr, const int* s_tok, const float* s_w) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hl = lane & 15, half = lane >> 4;
  const int nch = a.K / 32;
  const size_t crow = a.K / 2;
  const bool sh = te.group == a.E;
  const size_t e = sh ? 0 : static_cast<size_t>(te.group);
  const uint8_t* cd = (sh ? a.scodes0 : a.codes0) + e * a.N_out * crow;
  const uint16_t* sd = (sh ? a.sscale0 : a.scale0) + e * a.N_out * static_cast<size_t>(nch);
  constexpr int R = (NT <= 4 && MC <= 3) ? 4 : 2;  // rows per half-warp and pass
  constexpr int V = R * NT;
#pragma unroll 1
  for (int p = 0; p < kDownWarpRows / (2 * R); ++p) {
    const int j0 = jb + warp * kDownWarpRows + p * 2 * R + half * R;
    uint4 cw[R][MC];
    float sw[R][MC];
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int m = 0; m < MC; ++m) {
        cw[r][m] = ld_stream16(cd + static_cast<size_t>(j0 + r) * crow +
                               static_cast<size_t>(hl + 16 * m) * 16);
        sw[r][m] = bf16_bits_to_float(__ldg(sd + static_cast<size_t>(j0 + r) * nch + hl + 16 * m));
      }
    }
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
#pragma unroll
    for (int m = 0; m < MC; ++m) {
      const int c = hl + 16 * m;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t < nt) {
          const uint4* ap = s_act + static_cast<size_t>(t) * 4 * nch + c;
          const uint4 av[4] = {ap[0], ap[nch], ap[2 * nch], ap[3 * nch]};
          const float sig = s_sig[t * nch + c];
          const int corr = s_corr[t * nch + c];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int v = group_dot(cw[r][m], av, corr);
            acc[r * NT + t] = fmaf(static_cast<float>(v), sw[r][m] * sig, acc[r * NT + t]);
          }
        }
      }
    }
    const float val = reduce_scatter<V, 16>(acc, lane);
    constexpr int kLanesPerValue = 16 / V;
    const int idx = hl / kLanesPerValue;
    const int r = idx / NT, t = idx % NT;
    if (hl % kLanesPerValue == 0 && t < nt) {
      const int j = j0 + r;
      if (EPI == kEpiScatterAdd) {
        const int tok = s_tok[t];
        if (tok >= 0) atomicAdd(a.out + static_cast<size_t>(tok) * a.N_out + j, s_w[t] * val);
      } else {
        const int rr = te.row0 + t;
        if (rr < a.total_rows) a.out[static_cast<size_t>(rr) * a.N_out + j] = val;
      }
    }
  }
}

template <int MC, int EPI>
__global__ void __launch_bounds__(kThreads, 2) int4_gemv_down_kernel(const GemvArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int nch = a.K / 32;
  uint4* s_act = reinterpret_cast<uint4*>(smem);
  float* s_sig = reinterpret_cast<float*>(s_act + static_cast<size_t>(kRows) * 4 * nch);
  int* s_corr = reinterpret_cast<int*>(s_sig + kRows * nch);
  __shared__ int s_tok[kRows];
  __shared__ float s_w[kRows];

  pdl_wait();
  pdl_launch_dependents();
  const int nrb = a.N_out / kDownUnitRows;
  const int total = a.table[0] * nrb;
  int staged = -1;
  for (int u = blockIdx.x; u < total; u += gridDim.x) {
    const int ei = u / nrb, rb = u - ei * nrb;
    const TileEntry te = table_entry(a.table, ei);
    const int nt = min(te.nrows, kRows);
    if (ei != staged) {
      __syncthreads();  // every warp is done with the previous rows
      // the entry's h planes are laid out as in shared memory: a plain copy
      const size_t row_words = static_cast<size_t>(4) * nch;  // 16-byte words per row
      for (int i = threadIdx.x; i < nt * static_cast<int>(row_words); i += kThreads) {
        const int t = i / static_cast<int>(row_words);
        const int rr = te.row0 + t;
        s_act[i] = rr < a.total_rows
                       ? __ldcg(reinterpret_cast<const uint4*>(a.hq) + static_cast<size_t>(rr) * row_words +
                                (i - t * static_cast<int>(row_words)))
                       : make_uint4(0u, 0u, 0u, 0u);
      }
      for (int i = threadIdx.x; i < nt * nch; i += kThreads) {
        const int t = i / nch;
        const int rr = te.row0 + t;
        const size_t src = static_cast<size_t>(rr) * nch + (i - t * nch);
        s_sig[i] = rr < a.total_rows ? __ldcg(a.hs + src) : 0.f;
        s_corr[i] = rr < a.total_rows ? __ldcg(a.hc + src) : 0;
      }
      if (threadIdx.x < kRows) {
        const int r = te.row0 + threadIdx.x;
        int tok = -1;
        float w = 0.f;
        if (EPI == kEpiScatterAdd && threadIdx.x < nt && r < a.total_rows) {
          tok = a.gather[r];
          w = a.roww[r];
          if (tok < 0 || tok >= a.out_rows) tok = -1;
        }
        s_tok[threadIdx.x] = tok;
        s_w[threadIdx.x] = w;
      }
      __syncthreads();
      staged = ei;
    }
    const int jb = rb * kDownUnitRows;
    if (nt <= 1)
      down_unit<MC, 1, EPI>(a, te, jb, nt, s_act, s_sig, s_corr, s_tok, s_w);
    else if (nt <= 2)
      down_unit<MC, 2, EPI>(a, te, jb, nt, s_act, s_sig, s_corr, s_tok, s_w);
    else if (nt <= 4)
      down_unit<MC, 4, EPI>(a, te, jb, nt, s_act, s_sig, s_corr, s_tok, s_w);
    else
      down_unit<MC, 8, EPI>(a, te, jb, nt, s_act, s_sig, s_corr, s_tok, s_w);
  }
}

size_t act_smem_bytes(int K) { return static_cast<size_t>(kRows) * (K / 32) * (4 * 16 + 8); }

template <typename Kern>
cudaError_t launch_gemv(Kern kern, const GemvArgs& a, int grid, size_t smem, cudaStream_t s) {
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

GemvArgs args_of(const Int4GemvLaunch& L) {
  GemvArgs a{};
  a.table = L.table;
  a.E = L.E;
  a.K = L.K;
  a.N_out = L.N_out;
  a.total_rows = L.total_rows;
  a.out_rows = L.out_rows;
  a.x = L.x;
  a.xrows = L.xrows;
  a.codes0 = static_cast<const uint8_t*>(L.codes[0]);
  a.codes1 = static_cast<const uint8_t*>(L.codes[1]);
  a.scale0 = static_cast<const uint16_t*>(L.scale[0]);
  a.scale1 = static_cast<const uint16_t*>(L.scale[1]);
  a.scodes0 = static_cast<const uint8_t*>(L.scodes[0]);
  a.scodes1 = static_cast<const uint8_t*>(L.scodes[1]);
  a.sscale0 = static_cast<const uint16_t*>(L.sscale[0]);
  a.sscale1 = static_cast<const uint16_t*>(L.sscale[1]);
  a.hq = L.hq;
  a.hs = L.hs;
  a.hc = L.hc;
  a.gather = L.gather;
  a.roww = L.roww;
  a.out = L.out;
  return a;
}

}  // namespace

bool int4_gemv_shape_ok(int H, int I) {
  return H % 1024 == 0 && H <= 4096 && I % 512 == 0 && I <= 2048;
}

cudaError_t launch_int4_gemv_gateup(const Int4GemvLaunch& L, cudaStream_t s) {
  if (!int4_gemv_shape_ok(L.K, L.N_out) || L.grid <= 0) return cudaErrorInvalidValue;
  const GemvArgs a = args_of(L);
  const size_t smem = act_smem_bytes(L.K) + static_cast<size_t>(kRows) * kUnitFeatures * 4;
  switch (L.K / 1024) {
    case 1: return launch_gemv(int4_gemv_gateup_kernel<1>, a, L.grid, smem, s);
    case 2: return launch_gemv(int4_gemv_gateup_kernel<2>, a, L.grid, smem, s);
    case 3: return launch_gemv(int4_gemv_gateup_kernel<3>, a, L.grid, smem, s);
    default: return launch_gemv(int4_gemv_gateup_kernel<4>, a, L.grid, smem, s);
  }
}

cudaError_t launch_int4_gemv_down(const Int4GemvLaunch& L, cudaStream_t s) {
  if (!int4_gemv_shape_ok(L.N_out, L.K) || L.grid <= 0) return cudaErrorInvalidValue;
  const GemvArgs a = args_of(L);
  const size_t smem = act_smem_bytes(L.K);
  const bool add = L.epilogue == kEpiScatterAdd;
  switch (L.K / 512) {
    case 1:
      return add ? launch_gemv(int4_gemv_down_kernel<1, kEpiScatterAdd>, a, L.grid, smem, s)
                 : launch_gemv(int4_gemv_down_kernel<1, kEpiStoreRows>, a, L.grid, smem, s);
    case 2:
      return add ? launch_gemv(int4_gemv_down_kernel<2, kEpiScatterAdd>, a, L.grid, smem, s)
                 : launch_gemv(int4_gemv_down_kernel<2, kEpiStoreRows>, a, L.grid, smem, s);
    case 3:
      return add ? launch_gemv(int4_gemv_down_kernel<3, kEpiScatterAdd>, a, L.grid, smem, s)
                 : launch_gemv(int4_gemv_down_kernel<3, kEpiStoreRows>, a, L.grid, smem, s);
    default:
      return add ? launch_gemv(int4_gemv_down_kernel<4, kEpiScatterAdd>, a, L.grid, smem, s)
                 : launch_gemv(int4_gemv_down_kernel<4, kEpiStoreRows>, a, L.grid, smem, s);
  }
}

}  // namespace moe
