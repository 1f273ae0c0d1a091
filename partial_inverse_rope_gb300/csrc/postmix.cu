// Fused inverse RoPE + ungrouped VHA postmix on GB300 (sm_103a): forward and
// backward kernels, the fixed-order dM reduction, and their C-ABI launchers.
//
// Method: PaddleFleet PR #1772, "Fuse HCA inverse RoPE into the VHA postmix,
// and the sparse-attention KV index remap" -- English description item 1
// (rotation only on the trailing pe channels; the postmix is an [nh, nh] GEMM
// over heads, so channels are a pure N dimension), Chinese description
// section 1 (dM = sum_{t,c} dOut[t,h,c] * O_roped[t,h',c]) and the revision
// note (input gradient = postmix input gradient pushed back through the
// rotation).
//
// GB300 design (one persistent CTA per SM, warp-specialised):
//   * O (or dY) is viewed as a 2-D matrix [sq*nh, d]. A tile is R = P*nh rows
//     (P whole positions, R <= 128) by NC channels. TMA loads it into shared
//     memory as 64-channel, 128-byte-swizzled boxes.
//   * The head mix of P positions is ONE tcgen05 MMA chain with M = 128:
//     D[128 x NC] = A[128 x 128] * B[128 x NC], A = blockdiag_P(M) (or of M^T
//     for the input gradient) split into bf16 hi + lo terms, B = the tile.
//     Accumulation is fp32 in tensor memory (TMEM).
//   * Because the rotation depends only on the position, invrope(M . O) =
//     M . invrope(O): the epilogue rotates the fp32 accumulator's pe columns,
//     rounds once to bf16, writes the result into the tile's own shared
//     buffer and TMA-stores it. No rotated copy of O ever exists in HBM.
//   * Backward: the same chain on dY with M^T gives G, rotated by +a into dO.
//     In the same pass a second chain accumulates dY_tile . X_tile^T into a
//     persistent 128 x 128 TMEM accumulator, whose diagonal nh x nh blocks sum
//     to this CTA's share of dM. X = invrope(O) is exact bf16 on the nope
//     channels; on the pe channels it is split into hi + lo bf16 terms (hi
//     replaces O in place, lo goes to a side buffer) so dM carries ~16 bits.
//   * Every wait is bounded (about two seconds); a wait that runs out records
//     a fault code, raises a CTA-wide abort flag and the CTA winds down.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.h"
#include "ptx.cuh"

namespace invrope {

__device__ unsigned int g_fault_code = 0;

namespace {

constexpr int kRowsMax = 128;                            // MMA M = rows of a tile
constexpr int kChunkCols = 64;                           // channels per swizzle row
constexpr int kChunkBytes = kRowsMax * kChunkCols * 2;   // one 64-channel box, 16 KB
constexpr int kPosPerTileMax = 32;                       // caps the cos/sin table
constexpr int kMaxHalf = 32;                             // pe / 2 <= 32
constexpr uint64_t kWaitLimitNs = 2000000000ull;         // bounded waits: 2 s

// fault codes: role in bits 8-11, barrier kind in bits 0-7
enum : unsigned { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3, kRoleTransform = 4 };
enum : unsigned { kBarFull = 1, kBarEmpty, kBarAccFull, kBarAccEmpty, kBarXFull, kBarXEmpty,
                  kBarD2, kBarDone, kBarXGo };

template <bool BWD>
struct KCfg {
  static constexpr int NC = BWD ? 64 : 128;              // channels per tile
  static constexpr int kChunks = NC / kChunkCols;
  static constexpr int kStages = 4;
  static constexpr int kTensorTile = kChunks * kChunkBytes;
  static constexpr int kStageBytes = (BWD ? 2 : 1) * kTensorTile;
  static constexpr int kNumAcc = 4;
  static constexpr int kD2Col = kNumAcc * NC;            // dM accumulator column (bwd)
  static constexpr int kTmemCols = 512;
  static constexpr int kThreads = BWD ? 320 : 192;
  // shared-memory carve-up (bytes from the 1024-aligned base)
  static constexpr int kOffA = 0;                        // A hi: 2 K-blocks, then A lo
  static constexpr int kABytes = 4 * kChunkBytes;
  static constexpr int kOffStage = kOffA + kABytes;
  static constexpr int kOffXlo = kOffStage + kStages * kStageBytes;
  static constexpr int kXloBytes = BWD ? kChunkBytes : 0;
  static constexpr int kTabBytes = kPosPerTileMax * kMaxHalf * 8;
  static constexpr int kOffTabEpi = kOffXlo + kXloBytes;
  static constexpr int kOffTabXf = kOffTabEpi + kTabBytes;
  static constexpr int kOffFreq = kOffTabXf + (BWD ? kTabBytes : 0);
  static constexpr int kOffBars = kOffFreq + kMaxHalf * 8;
  static constexpr int kNumBars = 2 * kStages + 2 * kNumAcc + 5;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 32;  // tmem base, abort flag, 5 wait slots
  static constexpr int kSmemAlloc = kSmemBytes + 1024;   // slack to align the base
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
  static_assert(BWD ? (kD2Col + 128 <= kTmemCols) : (kNumAcc * NC <= kTmemCols), "TMEM budget");
};

struct PostmixParams {
  CUtensorMap tm_in0;  // fwd: O      bwd: dY
  CUtensorMap tm_in1;  // bwd: O
  CUtensorMap tm_out;  // fwd: Y      bwd: dO
  const float* M;
  float* ws;           // bwd: per-CTA dM partials [gridDim.x][nh][nh]
  int64_t sq;
  int64_t pos0;
  int64_t n_tiles;
  double theta;
  int nh, nope, pe, d;
  int P, R;            // positions and rows per tile
  int n_ct;            // channel tiles
};

struct Tile {
  int rt, ct, row0, c0, nch;
  int64_t s0;
  bool has_pe;
};

template <bool BWD>
__device__ __forceinline__ Tile decode_tile(const PostmixParams& p, int64_t t) {
  using C = KCfg<BWD>;
  Tile x;
  x.rt = static_cast<int>(t / p.n_ct);
  x.ct = static_cast<int>(t - static_cast<int64_t>(x.rt) * p.n_ct);
  x.row0 = x.rt * p.R;
  x.c0 = x.ct * C::NC;
  const int left = p.d - x.c0;
  x.nch = min(C::kChunks, (left + kChunkCols - 1) / kChunkCols);
  x.s0 = static_cast<int64_t>(x.rt) * p.P;
  x.has_pe = (p.nope / C::NC) == x.ct;
  return x;
}

__device__ __forceinline__ void record_fault(unsigned code, volatile int* abort_flag) {
  atomicCAS(&g_fault_code, 0u, code);
  *abort_flag = 1;
}

// Bounded wait on an mbarrier phase. Returns false when the CTA is aborting.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned code) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((n & 63u) == 0) {
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
        record_fault(code, abort_flag);
        return false;
      }
    }
  }
}

// One leader thread of a 128-thread group does the bounded wait; the whole
// group learns the outcome through `slot` and named barrier `bar_id`, so every
// member either proceeds or winds down together (no member is left waiting at
// a named barrier for a peer that gave up).
__device__ __forceinline__ bool group_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned code, bool leader, volatile int* slot,
                                           uint32_t bar_id) {
  if (leader) *slot = wait_bar(bar, parity, abort_flag, code) ? 1 : 0;
  ptx::named_bar_sync(bar_id, 128);
  return *slot != 0;
}

// cos/sin of a = pos * f_i for the P positions of a tile, i < half.
// The angle is reduced exactly in 64-bit fixed point: F[i] = f_i / (2 pi) * 2^64,
// pos * F[i] mod 2^64 is the fractional turn count; its top 32 bits give a
// turn in [-1/2, 1/2) that sincospif evaluates.
__device__ __forceinline__ void fill_rot_table(float2* tab, const uint64_t* F, int64_t pos_first,
                                               int P, int half, int tid, int nthr) {
  const int n = P * half;
  for (int k = tid; k < n; k += nthr) {
    const int pl = k / half;
    const int i = k - pl * half;
    const uint64_t turns = static_cast<uint64_t>(pos_first + pl) * F[i];
    const int32_t ti = static_cast<int32_t>(turns >> 32);
    const float tf = static_cast<float>(ti) * 2.3283064365386963e-10f;  // 2^-32
    float sn, cs;
    sincospif(2.0f * tf, &sn, &cs);
    tab[k] = make_float2(cs, sn);
  }
}

// byte address of the 16-byte unit holding channel `col` (tile-relative) of row r
__device__ __forceinline__ uint32_t swz_unit_addr(uint32_t tile, int r, int col) {
  const int chunk = col >> 6;
  const int unit = (col & 63) >> 3;
  return tile + chunk * kChunkBytes + r * 128 + ((unit ^ (r & 7)) << 4);
}

__device__ __forceinline__ void st_shared_b16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ uint16_t ld_shared_b16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.b16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
  __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&b);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

template <bool BWD>
__global__ void __launch_bounds__(KCfg<BWD>::kThreads, 1)
    postmix_kernel(const __grid_constant__ PostmixParams p) {
  using C = KCfg<BWD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int S = C::kStages;
  constexpr int NA = C::kNumAcc;

  auto bar_full = [&](int s) { return base + C::kOffBars + 8u * s; };
  auto bar_empty = [&](int s) { return base + C::kOffBars + 8u * (S + s); };
  auto bar_acc_full = [&](int a) { return base + C::kOffBars + 8u * (2 * S + a); };
  auto bar_acc_empty = [&](int a) { return base + C::kOffBars + 8u * (2 * S + NA + a); };
  const uint32_t bar_x_full = base + C::kOffBars + 8u * (2 * S + 2 * NA);
  const uint32_t bar_x_empty = bar_x_full + 8;
  const uint32_t bar_d2 = bar_x_full + 16;
  const uint32_t bar_done = bar_x_full + 24;
  const uint32_t bar_x_go = bar_x_full + 32;
  auto stage_addr = [&](int s) { return base + C::kOffStage + static_cast<uint32_t>(s) * C::kStageBytes; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 4);
  volatile int* slot_epi = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 8);
  volatile int* slot_d2 = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 12);
  volatile int* slot_xf_full = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 16);
  volatile int* slot_xf_empty = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 20);
  volatile int* slot_xf_go = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 24);
  uint64_t* F = reinterpret_cast<uint64_t*>(gbase + C::kOffFreq);
  const int half = p.pe >> 1;

  // ------------------------------------------------------------ setup
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(bar_full(s), 1);
      ptx::mbar_init(bar_empty(s), 1);
    }
    for (int a = 0; a < NA; ++a) {
      ptx::mbar_init(bar_acc_full(a), 1);
      ptx::mbar_init(bar_acc_empty(a), 128);
    }
    ptx::mbar_init(bar_x_full, 128);
    ptx::mbar_init(bar_x_empty, 1);
    ptx::mbar_init(bar_d2, 1);
    ptx::mbar_init(bar_done, 1);
    ptx::mbar_init(bar_x_go, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&p.tm_in0);
    ptx::prefetch_tmap(&p.tm_out);
    if (BWD) ptx::prefetch_tmap(&p.tm_in1);
  }
  if (warp == 1) {
    ptx::tmem_alloc(base + C::kOffMisc, C::kTmemCols);
    ptx::tmem_relinquish();
  }

  // A = blockdiag_P(M) (forward) or blockdiag_P(M^T) (backward), bf16 hi + lo,
  // K-major with 128-byte swizzle: element (i, j) of K-block j/64 sits in row i.
  for (int u = threadIdx.x; u < kRowsMax * 16; u += blockDim.x) {
    const int i = u >> 4;
    const int j0 = (u & 15) << 3;
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float v[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int j = j0 + 2 * q + t;
        float x = 0.f;
        if (i < p.R && j < p.R && (i / p.nh) == (j / p.nh)) {
          const int gi = i % p.nh, gj = j % p.nh;
          x = BWD ? __ldg(p.M + gj * p.nh + gi) : __ldg(p.M + gi * p.nh + gj);
        }
        v[t] = x;
      }
      hw[q] = ptx::pack_bf16x2(v[0], v[1]);
      lw[q] = ptx::pack_bf16x2(v[0] - ptx::bf16_lo_f32(hw[q]), v[1] - ptx::bf16_hi_f32(hw[q]));
    }
    const int kb = j0 >> 6;
    const int unit = (j0 & 63) >> 3;
    const uint32_t off = kb * kChunkBytes + i * 128 + ((unit ^ (i & 7)) << 4);
    ptx::st_shared_v4(base + C::kOffA + off, hw[0], hw[1], hw[2], hw[3]);
    ptx::st_shared_v4(base + C::kOffA + 2 * kChunkBytes + off, lw[0], lw[1], lw[2], lw[3]);
  }
  // Zero every stage (rows >= R are never loaded and must read as 0) and X_lo.
  for (uint32_t o = threadIdx.x * 16u; o < static_cast<uint32_t>(S * C::kStageBytes + C::kXloBytes);
       o += blockDim.x * 16u)
    ptx::st_shared_v4(base + C::kOffStage + o, 0u, 0u, 0u, 0u);
  if (threadIdx.x < half) {
    const double f = pow(p.theta, -2.0 * static_cast<double>(threadIdx.x) / p.pe);
    F[threadIdx.x] = __double2ull_rn(f * 0.15915494309189535 * 18446744073709551616.0);
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int64_t G = gridDim.x;
  const int64_t t_begin = p.n_tiles * blockIdx.x / G;
  const int64_t t_end = p.n_tiles * (blockIdx.x + 1) / G;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      int64_t i = 0;
      for (int64_t t = t_begin; t < t_end; ++t, ++i) {
        const int st = static_cast<int>(i % S);
        const uint32_t ph = static_cast<uint32_t>((i / S) & 1);
        if (!wait_bar(bar_empty(st), ph ^ 1u, abort_flag, (kRoleProducer << 8) | kBarEmpty)) break;
        const Tile x = decode_tile<BWD>(p, t);
        const uint32_t bytes = static_cast<uint32_t>(x.nch * p.R * 128 * (BWD ? 2 : 1));
        ptx::mbar_arrive_expect_tx(bar_full(st), bytes);
        const uint32_t sa = stage_addr(st);
        for (int k = 0; k < x.nch; ++k)
          ptx::tma_load_2d(sa + k * kChunkBytes, &p.tm_in0, x.c0 + k * kChunkCols, x.row0, bar_full(st));
        if (BWD)
          for (int k = 0; k < x.nch; ++k)
            ptx::tma_load_2d(sa + C::kTensorTile + k * kChunkBytes, &p.tm_in1, x.c0 + k * kChunkCols,
                             x.row0, bar_full(st));
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t nks = static_cast<uint32_t>((p.R + 15) / 16);
      uint32_t d2_started = 0;
      int npe = 0;
      int64_t i = 0;
      for (int64_t t = t_begin; t < t_end; ++t, ++i) {
        const int st = static_cast<int>(i % S);
        const uint32_t ph = static_cast<uint32_t>((i / S) & 1);
        const int acc = static_cast<int>(i % NA);
        const uint32_t aph = static_cast<uint32_t>((i / NA) & 1);
        if (!wait_bar(bar_full(st), ph, abort_flag, (kRoleMma << 8) | kBarFull)) break;
        const Tile x = decode_tile<BWD>(p, t);
        // The transform warps only see pe tiles; this thread has observed every
        // stage phase in order, so it tells them when the pe tile has landed.
        if (BWD && x.has_pe) ptx::mbar_arrive(bar_x_go);
        if (!wait_bar(bar_acc_empty(acc), aph ^ 1u, abort_flag, (kRoleMma << 8) | kBarAccEmpty)) break;
        ptx::tc_fence_after();
        const uint32_t sa = stage_addr(st);
        // head mix: D[acc] = A_hi * B + A_lo * B, B = the tile (MN-major, K = rows)
        const uint32_t d_acc = tmem_base + static_cast<uint32_t>(acc * C::NC);
        const uint32_t idesc_mix = ptx::idesc_bf16_f32(128, 64u * x.nch, false, true);
        for (uint32_t hl = 0; hl < 2; ++hl)
          for (uint32_t ks = 0; ks < nks; ++ks) {
            const uint64_t ad = ptx::smem_desc_sw128(
                base + C::kOffA + hl * 2 * kChunkBytes + (ks >> 2) * kChunkBytes + (ks & 3) * 32, 16, 1024);
            const uint64_t bd = ptx::smem_desc_sw128(sa + ks * 2048, kChunkBytes, 1024);
            ptx::tc_mma_ss(d_acc, ad, bd, idesc_mix, (hl | ks) != 0);
          }
        if (BWD && x.has_pe) {
          if (!wait_bar(bar_x_full, static_cast<uint32_t>(npe & 1), abort_flag, (kRoleMma << 8) | kBarXFull))
            break;
          ptx::tc_fence_after();
        }
        if (BWD) {
          // dM share: D2 += dY_tile * X_tile^T (both K-major, K = channels)
          const uint32_t d2 = tmem_base + C::kD2Col;
          const uint32_t idesc_dm = ptx::idesc_bf16_f32(128, 128, false, false);
          const uint32_t xa = sa + C::kTensorTile;
          for (int k = 0; k < x.nch; ++k)
            for (uint32_t kk = 0; kk < 4; ++kk) {
              const uint64_t ad = ptx::smem_desc_sw128(sa + k * kChunkBytes + kk * 32, 16, 1024);
              const uint64_t bd = ptx::smem_desc_sw128(xa + k * kChunkBytes + kk * 32, 16, 1024);
              ptx::tc_mma_ss(d2, ad, bd, idesc_dm, d2_started);
              d2_started = 1;
            }
          if (x.has_pe) {
            const int kpe = (p.nope - x.c0) / kChunkCols;
            for (uint32_t kk = 0; kk < 4; ++kk) {
              const uint64_t ad = ptx::smem_desc_sw128(sa + kpe * kChunkBytes + kk * 32, 16, 1024);
              const uint64_t bd = ptx::smem_desc_sw128(base + C::kOffXlo + kk * 32, 16, 1024);
              ptx::tc_mma_ss(d2, ad, bd, idesc_dm, 1);
            }
          }
        }
        ptx::tc_commit(bar_acc_full(acc));
        if (BWD && x.has_pe) {
          ptx::tc_commit(bar_x_empty);
          ++npe;
        }
      }
      if (BWD) ptx::tc_commit(bar_d2);
      ptx::tc_commit(bar_done);
      wait_bar(bar_done, 0, abort_flag, (kRoleMma << 8) | kBarDone);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ---------------------------------------------------------- epilogue
    const int e = threadIdx.x - 64;
    const uint32_t quad = static_cast<uint32_t>(warp & 3);
    const int r = static_cast<int>(quad * 32) + lane;
    const uint32_t lane_addr = (quad * 32u) << 16;
    const bool row_ok = r < p.R;
    const int pl = row_ok ? r / p.nh : 0;
    float2* tab = reinterpret_cast<float2*>(gbase + C::kOffTabEpi);
    const float sgn = BWD ? 1.f : -1.f;  // rope (+a) for dO, inverse rope (-a) for Y
    int st_prev = -1;
    int64_t i = 0;
    for (int64_t t = t_begin; t < t_end; ++t, ++i) {
      const int st = static_cast<int>(i % S);
      const int acc = static_cast<int>(i % NA);
      const uint32_t aph = static_cast<uint32_t>((i / NA) & 1);
      if (!group_wait(bar_acc_full(acc), aph, abort_flag, (kRoleEpilogue << 8) | kBarAccFull, e == 0,
                      slot_epi, 1))
        break;
      ptx::tc_fence_after();
      const Tile x = decode_tile<BWD>(p, t);
      if (x.has_pe) {
        fill_rot_table(tab, F, p.pos0 + x.s0, p.P, half, e, 128);
        ptx::named_bar_sync(1, 128);
      }
      const uint32_t out_tile = stage_addr(st);
      const uint32_t taddr = tmem_base + lane_addr + static_cast<uint32_t>(acc * C::NC);
      for (int j0 = 0; j0 < x.nch * kChunkCols; j0 += 32) {
        uint32_t v[32];
        ptx::tmem_ld_x32(taddr + j0, v);
        ptx::tmem_ld_wait(v);
        if (row_ok) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t w0 = ptx::pack_bf16x2(__uint_as_float(v[8 * u + 0]), __uint_as_float(v[8 * u + 1]));
            const uint32_t w1 = ptx::pack_bf16x2(__uint_as_float(v[8 * u + 2]), __uint_as_float(v[8 * u + 3]));
            const uint32_t w2 = ptx::pack_bf16x2(__uint_as_float(v[8 * u + 4]), __uint_as_float(v[8 * u + 5]));
            const uint32_t w3 = ptx::pack_bf16x2(__uint_as_float(v[8 * u + 6]), __uint_as_float(v[8 * u + 7]));
            ptx::st_shared_v4(swz_unit_addr(out_tile, r, j0 + 8 * u), w0, w1, w2, w3);
          }
        }
      }
      if (x.has_pe) {
        // rotate the pe pairs of the fp32 accumulator, then round once
        const int pcol = p.nope - x.c0;
        const float2* rt = tab + pl * half;
        if ((half & 7) == 0) {
          for (int i0 = 0; i0 < half; i0 += 8) {
            uint32_t a[8], b[8];
            ptx::tmem_ld_x8(taddr + pcol + i0, a);
            ptx::tmem_ld_x8(taddr + pcol + half + i0, b);
            ptx::tmem_ld_wait(a, b);
            if (row_ok) {
              uint32_t w1[4], w2[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                float y1[2], y2[2];
#pragma unroll
                for (int s2 = 0; s2 < 2; ++s2) {
                  const int k = 2 * q + s2;
                  const float2 cs = rt[i0 + k];
                  const float x1 = __uint_as_float(a[k]), x2 = __uint_as_float(b[k]);
                  y1[s2] = x1 * cs.x - sgn * x2 * cs.y;
                  y2[s2] = x2 * cs.x + sgn * x1 * cs.y;
                }
                w1[q] = ptx::pack_bf16x2(y1[0], y1[1]);
                w2[q] = ptx::pack_bf16x2(y2[0], y2[1]);
              }
              ptx::st_shared_v4(swz_unit_addr(out_tile, r, pcol + i0), w1[0], w1[1], w1[2], w1[3]);
              ptx::st_shared_v4(swz_unit_addr(out_tile, r, pcol + half + i0), w2[0], w2[1], w2[2], w2[3]);
            }
          }
        } else {
          for (int ii = 0; ii < half; ++ii) {
            uint32_t a, b;
            ptx::tmem_ld_x1(taddr + pcol + ii, a);
            ptx::tmem_ld_x1(taddr + pcol + half + ii, b);
            ptx::tmem_ld_wait(a, b);
            if (row_ok) {
              const float2 cs = rt[ii];
              const float x1 = __uint_as_float(a), x2 = __uint_as_float(b);
              const int c1 = pcol + ii, c2 = pcol + half + ii;
              st_shared_b16(swz_unit_addr(out_tile, r, c1) + (c1 & 7) * 2, bf16_bits(x1 * cs.x - sgn * x2 * cs.y));
              st_shared_b16(swz_unit_addr(out_tile, r, c2) + (c2 & 7) * 2, bf16_bits(x2 * cs.x + sgn * x1 * cs.y));
            }
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar_acc_empty(acc));
      ptx::fence_proxy_async_smem();
      ptx::named_bar_sync(1, 128);
      if (e == 0) {
        for (int k = 0; k < x.nch; ++k)
          ptx::tma_store_2d(&p.tm_out, out_tile + k * kChunkBytes, x.c0 + k * kChunkCols, x.row0);
        ptx::bulk_commit();
        if (st_prev >= 0) {
          ptx::bulk_wait_read<1>();
          ptx::mbar_arrive(bar_empty(st_prev));
        }
        st_prev = st;
      }
    }
    if (e == 0) ptx::bulk_wait<0>();
    if (BWD) {
      // this CTA's dM share: sum of the diagonal nh x nh blocks of D2
      if (group_wait(bar_d2, 0, abort_flag, (kRoleEpilogue << 8) | kBarD2, e == 0, slot_d2, 1)) {
        ptx::tc_fence_after();
        float* red = reinterpret_cast<float*>(gbase + C::kOffA);  // A is dead now
        const int lo = pl * p.nh;
        for (int j0 = 0; j0 < 128; j0 += 32) {
          uint32_t v[32];
          ptx::tmem_ld_x32(tmem_base + lane_addr + C::kD2Col + j0, v);
          ptx::tmem_ld_wait(v);
          if (row_ok) {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              const int j = j0 + jj;
              if (j >= lo && j < lo + p.nh) red[r * p.nh + (j - lo)] = __uint_as_float(v[jj]);
            }
          }
        }
        ptx::named_bar_sync(1, 128);
        const int nn = p.nh * p.nh;
        for (int idx = e; idx < nn; idx += 128) {
          const int g = idx / p.nh, h = idx - g * p.nh;
          float s = 0.f;
          for (int q = 0; q < p.P; ++q) s += red[(q * p.nh + g) * p.nh + h];
          p.ws[static_cast<int64_t>(blockIdx.x) * nn + idx] = s;
        }
      }
    }
  } else {
    // ---------------------------------------------------------- X = invrope(O) on the pe chunk (bwd)
    if (BWD) {
      const int xr = threadIdx.x - 192;
      float2* tab = reinterpret_cast<float2*>(gbase + C::kOffTabXf);
      int npe = 0;
      int64_t i = 0;
      for (int64_t t = t_begin; t < t_end; ++t, ++i) {
        const Tile x = decode_tile<BWD>(p, t);
        if (!x.has_pe) continue;
        const int st = static_cast<int>(i % S);
        const uint32_t ph = static_cast<uint32_t>((i / S) & 1);
        // Wait for the MMA thread's hand-off first: waiting on full[st] directly
        // could match a phase of the stage's previous tile (parity aliasing).
        if (!group_wait(bar_x_go, static_cast<uint32_t>(npe & 1), abort_flag, (kRoleTransform << 8) | kBarXGo,
                        xr == 0, slot_xf_go, 2))
          break;
        if (!group_wait(bar_full(st), ph, abort_flag, (kRoleTransform << 8) | kBarFull, xr == 0,
                        slot_xf_full, 2))
          break;
        if (!group_wait(bar_x_empty, static_cast<uint32_t>((npe & 1) ^ 1), abort_flag,
                        (kRoleTransform << 8) | kBarXEmpty, xr == 0, slot_xf_empty, 2))
          break;
        fill_rot_table(tab, F, p.pos0 + x.s0, p.P, half, xr, 128);
        ptx::named_bar_sync(2, 128);
        if (xr < p.R) {
          const int kpe = (p.nope - x.c0) / kChunkCols;
          const uint32_t oc = stage_addr(st) + C::kTensorTile + kpe * kChunkBytes;
          const uint32_t xl = base + C::kOffXlo;
          const int pc = p.nope - (x.c0 + kpe * kChunkCols);
          const float2* rt = tab + (xr / p.nh) * half;
          if ((half & 7) == 0) {
            for (int i0 = 0; i0 < half; i0 += 8) {
              const uint32_t a1 = swz_unit_addr(oc, xr, pc + i0);
              const uint32_t a2 = swz_unit_addr(oc, xr, pc + half + i0);
              uint32_t u1[4], u2[4];
              ptx::ld_shared_v4(a1, u1[0], u1[1], u1[2], u1[3]);
              ptx::ld_shared_v4(a2, u2[0], u2[1], u2[2], u2[3]);
              uint32_t h1[4], h2[4], l1[4], l2[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                float X1[2], X2[2];
#pragma unroll
                for (int s2 = 0; s2 < 2; ++s2) {
                  const float2 cs = rt[i0 + 2 * q + s2];
                  const float x1 = s2 ? ptx::bf16_hi_f32(u1[q]) : ptx::bf16_lo_f32(u1[q]);
                  const float x2 = s2 ? ptx::bf16_hi_f32(u2[q]) : ptx::bf16_lo_f32(u2[q]);
                  X1[s2] = x1 * cs.x + x2 * cs.y;
                  X2[s2] = x2 * cs.x - x1 * cs.y;
                }
                h1[q] = ptx::pack_bf16x2(X1[0], X1[1]);
                h2[q] = ptx::pack_bf16x2(X2[0], X2[1]);
                l1[q] = ptx::pack_bf16x2(X1[0] - ptx::bf16_lo_f32(h1[q]), X1[1] - ptx::bf16_hi_f32(h1[q]));
                l2[q] = ptx::pack_bf16x2(X2[0] - ptx::bf16_lo_f32(h2[q]), X2[1] - ptx::bf16_hi_f32(h2[q]));
              }
              ptx::st_shared_v4(a1, h1[0], h1[1], h1[2], h1[3]);
              ptx::st_shared_v4(a2, h2[0], h2[1], h2[2], h2[3]);
              ptx::st_shared_v4(swz_unit_addr(xl, xr, pc + i0), l1[0], l1[1], l1[2], l1[3]);
              ptx::st_shared_v4(swz_unit_addr(xl, xr, pc + half + i0), l2[0], l2[1], l2[2], l2[3]);
            }
          } else {
            for (int ii = 0; ii < half; ++ii) {
              const int c1 = pc + ii, c2 = pc + half + ii;
              const uint32_t a1 = swz_unit_addr(oc, xr, c1) + (c1 & 7) * 2;
              const uint32_t a2 = swz_unit_addr(oc, xr, c2) + (c2 & 7) * 2;
              const float x1 = bf16_bits_to_f32(ld_shared_b16(a1));
              const float x2 = bf16_bits_to_f32(ld_shared_b16(a2));
              const float2 cs = rt[ii];
              const float X1 = x1 * cs.x + x2 * cs.y, X2 = x2 * cs.x - x1 * cs.y;
              const uint16_t hb1 = bf16_bits(X1), hb2 = bf16_bits(X2);
              st_shared_b16(a1, hb1);
              st_shared_b16(a2, hb2);
              st_shared_b16(swz_unit_addr(xl, xr, c1) + (c1 & 7) * 2, bf16_bits(X1 - bf16_bits_to_f32(hb1)));
              st_shared_b16(swz_unit_addr(xl, xr, c2) + (c2 & 7) * 2, bf16_bits(X2 - bf16_bits_to_f32(hb2)));
            }
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(bar_x_full);
        ++npe;
      }
    }
  }

  // ------------------------------------------------------------ teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// dM[idx] = sum_c ws[c][idx] over the CTAs' partials in CTA order, with a
// compensated (Kahan) fp32 sum: deterministic and close to an fp64 sum.
__global__ void dm_reduce_kernel(const float* __restrict__ ws, float* __restrict__ dM, int nparts,
                                 int nn) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= nn) return;
  float s = 0.f, comp = 0.f;
  for (int c = 0; c < nparts; ++c) {
    const float y = ws[static_cast<int64_t>(c) * nn + idx] - comp;
    const float t = s + y;
    comp = (t - s) - y;
    s = t;
  }
  dM[idx] = s;
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D bf16 view [rows, d] with 64 x box_rows boxes, 128-byte swizzle.
bool make_tmap(CUtensorMap* m, const void* ptr, int64_t rows, int d, int box_rows) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kChunkCols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Shape {
  int P, R, n_ct;
  int64_t n_tiles;
};

int check_shape(int64_t sq, int nh, int nope, int pe, int nc, Shape* s) {
  if (sq < 0 || nh < 1 || nope < 0 || pe < 2 || (pe & 1)) return INVROPE_ERR_INVALID_ARG;
  const int64_t d = static_cast<int64_t>(nope) + pe;
  if (d % 8 != 0 || d > (1 << 20)) return INVROPE_ERR_INVALID_ARG;
  if (nh > 128) return INVROPE_ERR_UNSUPPORTED;
  if (nope / kChunkCols != (d - 1) / kChunkCols) return INVROPE_ERR_UNSUPPORTED;
  if (sq * nh >= (int64_t(1) << 31)) return INVROPE_ERR_UNSUPPORTED;
  s->P = 128 / nh < kPosPerTileMax ? 128 / nh : kPosPerTileMax;
  s->R = s->P * nh;
  s->n_ct = static_cast<int>((d + nc - 1) / nc);
  s->n_tiles = ((sq + s->P - 1) / s->P) * s->n_ct;
  return INVROPE_OK;
}

template <bool BWD>
int ensure_smem_attr(int device) {
  static std::mutex mu;
  static bool done[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return INVROPE_ERR_DEVICE;
  if (!done[device]) {
    const cudaError_t err = cudaFuncSetAttribute(postmix_kernel<BWD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 KCfg<BWD>::kSmemAlloc);
    if (err != cudaSuccess) return cuda_fail(err);
    done[device] = true;
  }
  return INVROPE_OK;
}

bool valid_theta(double theta) { return std::isfinite(theta) && theta > 0.0; }

}  // namespace

// Grid size of the backward kernel (one dM partial per CTA).
static int64_t bwd_grid(const Shape& s, int sms) { return s.n_tiles < sms ? s.n_tiles : sms; }

}  // namespace invrope

using namespace invrope;

extern "C" int invrope_postmix_fwd(const void* O, const float* M, void* Y, int64_t sq, int nh, int nope, int pe,
                                   int64_t pos0, double theta, struct CUstream_st* stream) {
  Shape s;
  int st = check_shape(sq, nh, nope, pe, KCfg<false>::NC, &s);
  if (st != INVROPE_OK) return st;
  if (pos0 < 0 || !valid_theta(theta)) return INVROPE_ERR_INVALID_ARG;
  if (sq == 0) return INVROPE_OK;
  if (!O || !M || !Y || !aligned(O, 16) || !aligned(Y, 16) || !aligned(M, 4)) return INVROPE_ERR_INVALID_ARG;
  const size_t tbytes = static_cast<size_t>(sq) * nh * (nope + pe) * 2;
  const size_t mbytes = static_cast<size_t>(nh) * nh * 4;
  if (overlaps(Y, tbytes, O, tbytes) || overlaps(Y, tbytes, M, mbytes)) return INVROPE_ERR_INVALID_ARG;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != INVROPE_OK) return st;
  if ((st = ensure_smem_attr<false>(dev.device)) != INVROPE_OK) return st;
  PostmixParams p;
  std::memset(&p, 0, sizeof(p));
  const int d = nope + pe;
  if (!make_tmap(&p.tm_in0, O, sq * nh, d, s.R) || !make_tmap(&p.tm_out, Y, sq * nh, d, s.R))
    return INVROPE_ERR_CUDA;
  p.tm_in1 = p.tm_in0;
  p.M = M;
  p.ws = nullptr;
  p.sq = sq;
  p.pos0 = pos0;
  p.n_tiles = s.n_tiles;
  p.theta = theta;
  p.nh = nh;
  p.nope = nope;
  p.pe = pe;
  p.d = d;
  p.P = s.P;
  p.R = s.R;
  p.n_ct = s.n_ct;
  const int64_t grid = s.n_tiles < dev.sms ? s.n_tiles : dev.sms;
  postmix_kernel<false><<<static_cast<unsigned>(grid), KCfg<false>::kThreads, KCfg<false>::kSmemAlloc,
                          reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return check_launch();
}

extern "C" size_t invrope_postmix_bwd_workspace_bytes(int64_t sq, int nh, int nope, int pe) {
  Shape s;
  if (check_shape(sq, nh, nope, pe, KCfg<true>::NC, &s) != INVROPE_OK) return 0;
  DeviceInfo dev;
  if (current_device(&dev) != INVROPE_OK) return 0;
  const int64_t grid = sq == 0 ? 1 : bwd_grid(s, dev.sms);
  return static_cast<size_t>(grid) * nh * nh * sizeof(float);
}

extern "C" int invrope_postmix_bwd(const void* dY, const void* O, const float* M, void* dO, float* dM,
                                   void* workspace, size_t workspace_bytes, int64_t sq, int nh, int nope, int pe,
                                   int64_t pos0, double theta, struct CUstream_st* stream) {
  Shape s;
  int st = check_shape(sq, nh, nope, pe, KCfg<true>::NC, &s);
  if (st != INVROPE_OK) return st;
  if (pos0 < 0 || !valid_theta(theta)) return INVROPE_ERR_INVALID_ARG;
  if (!M || !dM || !aligned(M, 4) || !aligned(dM, 4)) return INVROPE_ERR_INVALID_ARG;
  if (sq > 0 && (!dY || !O || !dO || !aligned(dY, 16) || !aligned(O, 16) || !aligned(dO, 16)))
    return INVROPE_ERR_INVALID_ARG;
  const size_t tbytes = static_cast<size_t>(sq) * nh * (nope + pe) * 2;
  const size_t mbytes = static_cast<size_t>(nh) * nh * 4;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != INVROPE_OK) return st;
  const int64_t grid = sq == 0 ? 0 : bwd_grid(s, dev.sms);
  const size_t need = static_cast<size_t>(grid == 0 ? 1 : grid) * nh * nh * sizeof(float);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return INVROPE_ERR_WORKSPACE;
  if (overlaps(dO, tbytes, dY, tbytes) || overlaps(dO, tbytes, O, tbytes) || overlaps(dO, tbytes, M, mbytes) ||
      overlaps(dM, mbytes, dY, tbytes) || overlaps(dM, mbytes, O, tbytes) || overlaps(dM, mbytes, M, mbytes) ||
      overlaps(dM, mbytes, dO, tbytes) || overlaps(workspace, need, dY, tbytes) ||
      overlaps(workspace, need, O, tbytes) || overlaps(workspace, need, M, mbytes) ||
      overlaps(workspace, need, dO, tbytes) || overlaps(workspace, need, dM, mbytes))
    return INVROPE_ERR_INVALID_ARG;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int nn = nh * nh;
  if (grid > 0) {
    if ((st = ensure_smem_attr<true>(dev.device)) != INVROPE_OK) return st;
    PostmixParams p;
    std::memset(&p, 0, sizeof(p));
    const int d = nope + pe;
    if (!make_tmap(&p.tm_in0, dY, sq * nh, d, s.R) || !make_tmap(&p.tm_in1, O, sq * nh, d, s.R) ||
        !make_tmap(&p.tm_out, dO, sq * nh, d, s.R))
      return INVROPE_ERR_CUDA;
    p.M = M;
    p.ws = static_cast<float*>(workspace);
    p.sq = sq;
    p.pos0 = pos0;
    p.n_tiles = s.n_tiles;
    p.theta = theta;
    p.nh = nh;
    p.nope = nope;
    p.pe = pe;
    p.d = d;
    p.P = s.P;
    p.R = s.R;
    p.n_ct = s.n_ct;
    postmix_kernel<true><<<static_cast<unsigned>(grid), KCfg<true>::kThreads, KCfg<true>::kSmemAlloc, cs>>>(p);
    if ((st = check_launch()) != INVROPE_OK) return st;
  }
  dm_reduce_kernel<<<(nn + 127) / 128, 128, 0, cs>>>(static_cast<const float*>(workspace), dM,
                                                     static_cast<int>(grid), nn);
  return check_launch();
}

extern "C" int invrope_take_device_fault(int* fault) {
  if (!fault) return INVROPE_ERR_INVALID_ARG;
  cudaError_t err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return cuda_fail(err);
  unsigned v = 0;
  if ((err = cudaMemcpyFromSymbol(&v, g_fault_code, sizeof(v))) != cudaSuccess) return cuda_fail(err);
  const unsigned zero = 0;
  if ((err = cudaMemcpyToSymbol(g_fault_code, &zero, sizeof(zero))) != cudaSuccess) return cuda_fail(err);
  *fault = static_cast<int>(v);
  return INVROPE_OK;
}
