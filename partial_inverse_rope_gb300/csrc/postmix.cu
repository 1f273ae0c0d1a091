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
//     128 x 128 TMEM accumulator, whose diagonal nh x nh blocks sum to this
//     CTA's share of dM (the stacked kernel below: one M = 64 MMA per position
//     into a 64 x 64 accumulator that holds the position sum itself). Every
//     backward shape but the stacked one and tiny ones uses 128-channel tiles. X = invrope(O) is exact bf16 on the nope
//     channels; on the pe channels it is split into hi + lo bf16 terms (hi
//     replaces O in place, lo goes to a side buffer) so dM carries ~16 bits.
//   * Backward with nh = 64 and the pe block filling one 64-channel chunk
//     (e.g. 448 + 64): the head mix is instead one chain of four M = 128,
//     N = 128 MMAs. A = [M^T_hi ; M^T_lo] stacks the two bf16 terms along M
//     (rows 0-63 hi, 64-127 lo, K = the 64 heads) and B spans both positions
//     of the tile along N: its second 64-wide N block is the tile's rows
//     64-127, reached through the descriptor's N-block stride. The epilogue
//     adds the lo rows to the hi rows; the lo rows pass through the output
//     buffer as bf16, a rounding of about 2^-9 of a term that is itself about
//     2^-9 of the result. This is a quarter of the block-diagonal form's MMA
//     issue, with none of its zero blocks.
//   * Every wait is bounded (about two seconds); a wait that runs out records
//     a fault code, raises a CTA-wide abort flag and the CTA winds down.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace invrope {

__device__ unsigned int g_fault_code = 0;

// Debug-bounds builds (-DINVROPE_DEBUG_BOUNDS, see build.py --debug-bounds)
// check index invariants on the device and record 0xDB00 | id in the fault
// code when one fails, without trapping (the access itself still happens, so
// a check guards against silent corruption, not against a fault). In normal
// builds the checks compile to nothing.
#ifdef INVROPE_DEBUG_BOUNDS
#define INVROPE_DBG_CHECK(cond, id)                              \
  do {                                                           \
    if (!(cond)) atomicCAS(&g_fault_code, 0u, 0xDB00u | (id));   \
  } while (0)
#else
#define INVROPE_DBG_CHECK(cond, id) \
  do {                              \
  } while (0)
#endif

// Dynamic tile scheduling of the forward: one work-counter slot per launch
// (sched.cuh): the first tile of a CTA is its block index, later ones are
// claimed from the slot's counter.
__device__ SchedSlot g_sched[kSchedSlots];

namespace {

constexpr int kRowsMax = 128;                            // MMA M = rows of a tile
constexpr int kChunkCols = 64;                           // channels per swizzle row
constexpr int kChunkBytes = kRowsMax * kChunkCols * 2;   // one 64-channel box, 16 KB
constexpr int kPosPerTileMax = 32;     // caps the cos/sin tables (backward with pair blocks)
constexpr int kPosPerTileMaxFwd = 64;  // every other build (forward: one table; backward: one X_lo box)
constexpr int kMaxHalf = 32;                             // pe / 2 <= 32
constexpr uint64_t kWaitLimitNs = 2000000000ull;         // bounded waits: 2 s

// fault codes: role in bits 8-11, barrier kind in bits 0-7
enum : unsigned { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3, kRoleTransform = 4, kRoleStore = 5 };
enum : unsigned { kBarFull = 1, kBarEmpty, kBarAccFull, kBarAccEmpty, kBarXFull, kBarXEmpty,
                  kBarD2, kBarDone, kBarXGo, kBarOut, kBarM, kBarSeg, kBarD2Empty };

// WIDE (every backward shape but the stacked one and tiny ones): 128-channel
// tiles, so each head-mix MMA has N = 128 and a tile needs half as many of them.
// STK (backward, nh = 64, pe block = one whole chunk): the stacked head mix.
// Its dM share sums the tile's two positions in the MMAs themselves (M = 64
// per position, one 64 x 64 accumulator), so two D2 buffers take 128 TMEM
// columns (the drain of one segment overlaps the next segment's dM chains),
// with A in TMEM as in the other kernels. Two output buffers measured ~1 us
// faster than three, and a fifth input stage (the shared memory allows it)
// ~2 us slower, at the production shard.
// PAIRS: the build handles the general tiling's pair blocks (the forward, and
// the 128-channel backward built with them); those need a second X_lo box, so
// the backward builds without them have room for 64-position rotation tables.
template <bool BWD, bool WIDE = false, bool STK = false, bool PAIRS = !BWD || WIDE>
struct KCfg {
  static_assert(!STK || (BWD && !WIDE), "the stacked mix is a 64-channel backward");
  static constexpr int NC = (BWD && !WIDE) ? 64 : 128;   // channels per tile
  static constexpr int kChunks = NC / kChunkCols;
  static constexpr int kTensorTile = kChunks * kChunkBytes;
  static constexpr int kStageBytes = (BWD ? 2 : 1) * kTensorTile;   // input ring entry
  static constexpr int kStages = WIDE ? 2 : 4;           // input ring (bytes in flight alike)
  static constexpr int kOutBufs = BWD ? (STK ? 2 : 3) : 5;  // output ring of 64-channel chunks
  // TMA stores left reading shared memory (two buffers: one, waited after each store)
  static constexpr int kOutInflight = kOutBufs > 3 ? kOutBufs - 2 : 1;
  static constexpr int kNumAcc = BWD ? (WIDE ? 2 : 4) : 3;
  static constexpr int kNumD2 = STK ? 2 : 1;
  // TMEM columns: accumulators, then dM (bwd: one 128-column buffer, or two of
  // 64 columns for STK), then A hi (64) and A lo (64) (STK: 32 columns)
  static constexpr int kD2Col = kNumAcc * NC;
  static constexpr int kD2Cols = STK ? 64 : 128;
  static constexpr int kACol = 384;
  static constexpr int kTmemCols = 512;
  // warps: 0 TMA producer, 1 MMA issuer, 2-5 epilogue, (6-9 transform,) last = TMA store
  static constexpr int kWarpStore = BWD ? 10 : 6;
  static constexpr int kThreads = (kWarpStore + 1) * 32;
  // shared-memory carve-up (bytes from the 1024-aligned base)
  static constexpr int kOffStage = 0;
  static constexpr int kOffOut = kOffStage + kStages * kStageBytes;
  static constexpr int kOffXlo = kOffOut + kOutBufs * kChunkBytes;
  static constexpr int kXloBytes = BWD ? (PAIRS ? kChunks : 1) * kChunkBytes : 0;
  // bwd, stacked mix: fp32 exchange rows between the epilogue warp pairs (64 x 256 B)
  static constexpr int kOffXch = kOffXlo + kXloBytes;
  static constexpr int kXchBytes = STK ? 64 * 256 : 0;
  // rotation tables: positions per tile x 32 pairs (STK: 2 positions)
  static constexpr int kTabBytes = (STK ? 2 : (BWD && PAIRS) ? kPosPerTileMax : kPosPerTileMaxFwd) * kMaxHalf * 8;
  static constexpr int kOffTabEpi = kOffXch + kXchBytes;
  static constexpr int kOffTabXf = kOffTabEpi + kTabBytes;
  static constexpr int kOffFreq = kOffTabXf + (BWD ? kTabBytes : 0);
  static constexpr int kOffBars = kOffFreq + kMaxHalf * 8;
  // + backward: segment ring (4 full, 4 empty), D2 hand-back, second D2 pair
  static constexpr int kNumBars = 2 * kStages + 2 * kOutBufs + 2 * kNumAcc + 6 + (BWD ? 11 : 0);
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  // tmem base, abort flag, wait slots, tile ids (192 B), backward segment ring
  // and its broadcast slots (128 B)
  static constexpr int kSmemBytes = kOffMisc + 192 + (BWD ? 128 : 0);
  static constexpr int kSmemAlloc = kSmemBytes + 1024;   // slack to align the base
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
  static_assert(kNumAcc * NC + (BWD ? kNumD2 * kD2Cols : 0) <= kACol, "TMEM budget");
  static_assert(kStages * kStageBytes >= 128 * 129 * 4, "dM partial reduction reuses the input ring");
  static_assert(kOutInflight >= 1, "at least one store in flight");
  // the forward's bulk copy of M lands in the output ring and the buffers
  // after it (the backward copies M only when it fits in the ring itself)
  static_assert(BWD || kOffFreq - kOffOut >= 128 * 128 * 4, "M is copied into the output ring and the buffers after it");
};

struct PostmixParams {
  CUtensorMap tm_in0;  // fwd: O      bwd: dY   (general tiling: clipped at channel nope)
  CUtensorMap tm_in1;  // bwd: O                (general tiling: clipped at channel nope)
  CUtensorMap tm_out;  // fwd: Y      bwd: dO   (general tiling: clipped at channel nope)
  CUtensorMap tm_in0_pe;  // general tiling, pe tiles: in0 over all d channels
  CUtensorMap tm_in1_pe;  // general tiling, pe tiles: in1 over all d channels
  uint16_t* out;       // Y or dO (bf16 bits): the general tiling's pe tiles store directly
  const float* M;
  float* ws;           // bwd: per-CTA dM partials [gridDim.x][nh][nh]
  SchedSlot* sched;    // fwd: this launch's work-counter slot
  uint64_t F[kMaxHalf];  // rotary frequencies in turns per position, 0.64 fixed point
  int64_t sq;
  int64_t pos0;
  int64_t n_tiles;
  double theta;
  int nh, nope, pe, d;
  int P, R;            // positions and rows per tile
  int n_ct;            // channel tiles
  int stacked;         // bwd, nh = 64, pe block = one whole chunk: stacked head mix (below)
  const int32_t* pos;  // per-row positions (pos0 is added), or null: row s sits at pos0 + s
  int gs;              // heads per group of the head mix (nh: one [nh, nh] matrix)
  int m_bulk;          // M is copied into shared memory by one bulk copy at start (if it fits)
  // General tiling (the pe block does not lie inside one 64-channel box): channel
  // tiles [0, n_nope_ct) cover channels [0, nope & ~7) through the clipped maps;
  // tile n_nope_ct + j is pair block j, rotation pairs [32 j, 32 j + 32) of the
  // pe block, loaded as two boxes (first and second halves of its pairs).
  int gen;
  int n_nope_ct;
  int64_t rows;        // sq * nh: rows of the [sq*nh, d] view
  double log2_theta;   // rotary frequencies beyond the first 32 pairs are formed on the device
  // Backward schedule: CTA c first runs tiles [n_static c / G, n_static (c+1) / G)
  // into dM partial slot c; the tiles from n_static on form n_tail fixed blocks
  // (tail_na of tail_ba tiles, tail_nb of tail_bb tiles, then blocks of tail_bc
  // tiles), claimed one at a time from the launch's counter slot, block b into
  // partial slot G + b.
  int64_t n_static;
  int n_tail, tail_na, tail_ba, tail_nb, tail_bb, tail_bc;
};

// kind 0: a tile of the regular tiling (channels c0 + 64 k, TMA-stored);
// kind 1: a nope tile of the general tiling: channels [0, nope & ~7) through
//   the maps clipped there (a clip on a 16-byte boundary), TMA-stored;
// kind 2: a pair block of the general tiling: box 0 at channel xa holds the
//   first halves of pairs [32 j, 32 j + np), box 1 at channel xb their second
//   halves; its outputs are stored directly, pair by pair. Pair block 0 also
//   owns the nope channels [nope & ~7, nope), the first columns of its box 0.
struct Tile {
  int rt, ct, row0, c0, nch;
  int64_t s0;
  bool has_pe;
  int kind, xa, xb, j, np;
};

// channel of the first column of box k of a tile
__device__ __forceinline__ int box_x(const Tile& x, int k) { return k == 0 ? x.xa : x.xb; }

// Tile (rt, ct): row tile rt, channel tile ct.
template <bool BWD, bool WIDE = false, bool GEN = true>
__device__ __forceinline__ Tile make_tile(const PostmixParams& p, int rt, int ct) {
  using C = KCfg<BWD, WIDE>;
  Tile x;
  x.rt = rt;
  x.ct = ct;
  x.row0 = x.rt * p.R;
  x.s0 = static_cast<int64_t>(x.rt) * p.P;
  x.j = 0;
  x.np = 0;
  // the general tiling occurs in the forward and the 128-channel backward only
  // (GEN: the instantiation that takes it)
  constexpr bool kGen = (!BWD || WIDE) && GEN;
  const bool gen = kGen && p.gen;
  if (!gen || ct < p.n_nope_ct) {
    x.c0 = x.ct * C::NC;
    const int left = (gen ? (p.nope & ~7) : p.d) - x.c0;
    x.nch = min(C::kChunks, (left + kChunkCols - 1) / kChunkCols);
    x.has_pe = !gen && (p.nope / C::NC) == x.ct;
    x.kind = gen ? 1 : 0;
    x.xa = x.c0;
    x.xb = x.c0 + kChunkCols;
  } else {
    const int half = p.pe >> 1;
    x.j = ct - p.n_nope_ct;
    x.np = min(32, half - 32 * x.j);
    x.xa = (p.nope + 32 * x.j) & ~7;
    x.xb = (p.nope + half + 32 * x.j) & ~7;
    x.c0 = x.xa;
    x.nch = 2;
    x.has_pe = true;
    x.kind = 2;
  }
  return x;
}

// Tile t of the row-major (row tile, channel tile) order.
template <bool BWD, bool WIDE = false, bool GEN = true>
__device__ __forceinline__ Tile decode_tile(const PostmixParams& p, int64_t t) {
  // 32-bit division: the host guarantees n_tiles < 2^31 (64-bit division here
  // sits on the MMA issuer's critical path once per tile and is slow)
  const uint32_t tu = static_cast<uint32_t>(t);
  const uint32_t rt = tu / static_cast<uint32_t>(p.n_ct);
  return make_tile<BWD, WIDE, GEN>(p, static_cast<int>(rt), static_cast<int>(tu - rt * static_cast<uint32_t>(p.n_ct)));
}

__device__ __forceinline__ void record_fault(unsigned code, volatile int* abort_flag) {
  atomicCAS(&g_fault_code, 0u, code);
  *abort_flag = 1;
}

// Bounded wait on an mbarrier phase. Returns false when the CTA is aborting.
__device__ __forceinline__ bool wait_bar_for(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned code, uint64_t limit_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((n & 63u) == 0) {
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > limit_ns) {
        record_fault(code, abort_flag);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned code) {
  return wait_bar_for(bar, parity, abort_flag, code, kWaitLimitNs);
}

// Bounded wait that ignores the abort flag: for completions that must land
// before the CTA frees what they write to (in-flight MMAs, a bulk copy).
__device__ __forceinline__ bool wait_bar_noabort(uint32_t bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity))
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

// One thread waits for phase 0 of an mbarrier that nothing ever arrives on:
// the bounded wait must give up after limit_ns and record the self-test code.
__global__ void watchdog_selftest_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    wait_bar_for(ptx::smem_u32(&bar), 0, &abort_flag, INVROPE_WATCHDOG_SELFTEST_CODE, limit_ns);
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

// cos/sin of a = pos * f_i for the P positions of the tile starting at row
// s0, i < half. The position of row s is pos0 + s, or pos0 + pos[s] when a
// positions array is given (rows past sq, which are never stored, take pos0).
// The angle is reduced exactly in 64-bit fixed point: F[i] = f_i / (2 pi) * 2^64,
// pos * F[i] mod 2^64 is the fractional turn count (two's complement, so a
// negative position works too); its top 32 bits give an angle in [-pi, pi),
// where the hardware sine / cosine (__sincosf) is accurate to 2^-21.4
// absolute, far below the bf16 rounding of the outputs.
__device__ __forceinline__ void fill_rot_table(float2* tab, const uint64_t* F, const PostmixParams& p,
                                               int64_t s0, int half, int tid, int nthr) {
  const int n = p.P * half;
  const bool half32 = half == 32;  // the common pe = 64: no division
  for (int k = tid; k < n; k += nthr) {
    const int pl = half32 ? (k >> 5) : k / half;
    const int i = k - pl * half;
    const int64_t s = s0 + pl;
    const int64_t rel = p.pos ? (s < p.sq ? static_cast<int64_t>(__ldg(p.pos + s)) : 0) : s;
    const uint64_t turns = static_cast<uint64_t>(p.pos0 + rel) * F[i];
    const int32_t ti = static_cast<int32_t>(turns >> 32);
    const float tf = static_cast<float>(ti) * 2.3283064365386963e-10f;  // turns, 2^-32 units
    float sn, cs;
    __sincosf(6.28318530717958648f * tf, &sn, &cs);
    tab[k] = make_float2(cs, sn);
  }
}

// Rotary frequency of pair i as turns per position in 0.64 fixed point, formed
// on the device (pairs beyond the first 32, whose values the host does not pass).
__device__ __forceinline__ uint64_t freq_turns_fixed(int i, int pe, double log2_theta) {
  const double f = exp2(-2.0 * static_cast<double>(i) / static_cast<double>(pe) * log2_theta);
  return static_cast<uint64_t>(llrint(ldexp(f * 0.15915494309189535, 63))) << 1;
}

// The general tiling's pair block j: cos/sin of pairs 32 j + ii (ii < np) for
// the P positions of the tile starting at row s0, entry pl * 32 + ii.
__device__ __forceinline__ void fill_rot_table_gen(float2* tab, const uint64_t* F, const PostmixParams& p,
                                                   int64_t s0, int j, int np, int tid, int nthr) {
  const int n = p.P * 32;
  for (int k = tid; k < n; k += nthr) {
    const int pl = k >> 5, ii = k & 31;
    if (ii >= np) continue;
    const int i = 32 * j + ii;
    const uint64_t Fi = i < kMaxHalf ? F[i] : freq_turns_fixed(i, p.pe, p.log2_theta);
    const int64_t s = s0 + pl;
    const int64_t rel = p.pos ? (s < p.sq ? static_cast<int64_t>(__ldg(p.pos + s)) : 0) : s;
    const uint64_t turns = static_cast<uint64_t>(p.pos0 + rel) * Fi;
    const int32_t ti = static_cast<int32_t>(turns >> 32);
    const float tf = static_cast<float>(ti) * 2.3283064365386963e-10f;
    float sn, cs;
    __sincosf(6.28318530717958648f * tf, &sn, &cs);
    tab[k] = make_float2(cs, sn);
  }
}

// byte address of the 16-byte unit holding channel `col` (tile-relative) of row r
__device__ __forceinline__ uint32_t swz_unit_addr(uint32_t tile, int r, int col) {
  INVROPE_DBG_CHECK(r >= 0 && r < kRowsMax && col >= 0 && col < 2 * kChunkCols, 1);
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

// One row or one column of the [nh, nh] head mix in its block-diagonal form
// (a grouped mix, p.M = [nh/gs, gs, gs], is zero between groups), read from
// p.M directly: it is a few KB and stays in L2 after the first thread block.
struct MixLine {
  const float* M;
  int gs, b, f;  // group size; first head of the fixed index's group; fixed index - b
  bool row;      // true: M[fixed][x]; false: M[x][fixed]
  __device__ __forceinline__ MixLine(const PostmixParams& p, int fixed, bool is_row)
      : M(p.M), gs(p.gs), row(is_row) {
    b = (fixed / p.gs) * p.gs;
    f = fixed - b;
  }
  __device__ __forceinline__ float at(int x) const {  // 0 <= x < nh
    const unsigned o = static_cast<unsigned>(x - b);
    if (o >= static_cast<unsigned>(gs)) return 0.f;
    return __ldg(M + static_cast<int64_t>(b) * gs + (row ? f * gs + static_cast<int>(o) : static_cast<int>(o) * gs + f));
  }
};

template <bool BWD, bool WIDE = false, bool STK = false, bool GEN = true>
__global__ void __launch_bounds__(KCfg<BWD, WIDE, STK, (!BWD || WIDE) && GEN>::kThreads, 1)
    postmix_kernel(const __grid_constant__ PostmixParams p) {
  using C = KCfg<BWD, WIDE, STK, (!BWD || WIDE) && GEN>;
  // the general tiling's pair blocks occur in the forward and the 128-channel backward only
  constexpr bool kGen = (!BWD || WIDE) && GEN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int S = C::kStages;
  constexpr int OB = C::kOutBufs;
  constexpr int NA = C::kNumAcc;

  auto bar_full = [&](int s) { return base + C::kOffBars + 8u * s; };
  auto bar_empty = [&](int s) { return base + C::kOffBars + 8u * (S + s); };
  auto bar_ob_full = [&](int b) { return base + C::kOffBars + 8u * (2 * S + b); };
  auto bar_ob_empty = [&](int b) { return base + C::kOffBars + 8u * (2 * S + OB + b); };
  auto bar_acc_full = [&](int a) { return base + C::kOffBars + 8u * (2 * S + 2 * OB + a); };
  auto bar_acc_empty = [&](int a) { return base + C::kOffBars + 8u * (2 * S + 2 * OB + NA + a); };
  const uint32_t bar_x_full = base + C::kOffBars + 8u * (2 * S + 2 * OB + 2 * NA);
  const uint32_t bar_x_empty = bar_x_full + 8;
  const uint32_t bar_d2 = bar_x_full + 16;
  const uint32_t bar_done = bar_x_full + 24;
  const uint32_t bar_x_go = bar_x_full + 32;
  const uint32_t bar_m = bar_x_full + 40;  // M's bulk copy into shared memory
  // backward: segment ring (full: the producer published segment k; empty: its
  // four consumers have read it) and D2 handed back by the drain
  auto bar_seg_full = [&](int k) { return bar_x_full + 48 + 8u * k; };
  auto bar_seg_empty = [&](int k) { return bar_x_full + 80 + 8u * k; };
  const uint32_t bar_d2_empty = bar_x_full + 112;
  // D2 buffer b: full (the segment's last dM MMA completed) and empty (drained)
  auto bar_d2f = [&](int b) { return b ? bar_x_full + 120 : bar_d2; };
  auto bar_d2e = [&](int b) { return b ? bar_x_full + 128 : bar_d2_empty; };
  auto stage_addr = [&](int s) { return base + C::kOffStage + static_cast<uint32_t>(s) * C::kStageBytes; };
  auto out_addr = [&](int b) { return base + C::kOffOut + static_cast<uint32_t>(b) * kChunkBytes; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 4);
  volatile int* slot_epi = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 8);   // [2]
  volatile int* slot_ob = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 16);   // [2]
  volatile int* slot_d2 = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 24);
  volatile int* slot_xf_full = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 28);
  volatile int* slot_xf_empty = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 32);
  volatile int* slot_xf_go = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 36);
  // forward: tile ids handed from role to role (-1 = no more tiles)
  volatile int* stage_tile = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 64);  // [S]
  volatile int* acc_tile = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 96);    // [NA]
  volatile int* ob_tile = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 128);    // [OB]
  volatile int* ob_chunk = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 160);   // [OB]
  static_assert(S <= 8 && NA <= 8 && OB <= 8, "tile-id slots");
  // backward segment ring: entry k = {t0, t1, slot} (t0 < 0: no more segments),
  // and per-group broadcast slots {ok, t0, t1, slot} for the epilogue and the
  // transform warps (two each, alternating by segment parity)
  volatile int* seg_ring = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 192);   // [4][4]
  volatile int* seg_bc_epi = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 256);  // [2][4]
  volatile int* seg_bc_xf = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 288);   // [2][4]
  uint64_t* F = reinterpret_cast<uint64_t*>(gbase + C::kOffFreq);
  const int half = p.pe >> 1;
  // Accumulator ring: NA accumulators of NC columns, or 2 of 128 columns for the
  // stacked backward mix (the same 256 TMEM columns).
  constexpr bool stk = STK;
  static_assert(!BWD || NA == 4 || NA == 2, "the backward ring is indexed with shifts");
  const uint32_t na_sh = (stk || NA == 2) ? 1u : 2u;
  const uint32_t acc_cols = stk ? 128u : static_cast<uint32_t>(C::NC);
  auto acc_of = [&](uint32_t i) { return static_cast<int>(BWD ? i & ((1u << na_sh) - 1u) : i % NA); };
  auto acc_phase = [&](uint32_t i) { return BWD ? (i >> na_sh) & 1u : (i / NA) & 1u; };

  // one input tile into stage st: its full barrier expects the bytes, then the
  // 64-channel boxes (and, backward, O's boxes behind dY's)
  auto load_tile = [&](int st, int64_t t) {
    const Tile x = decode_tile<BWD, WIDE, GEN>(p, t);
    INVROPE_DBG_CHECK(t >= 0 && t < p.n_tiles && x.row0 >= 0 && x.xa % 8 == 0 && x.xa < p.d &&
                          (x.nch < 2 || (x.xb % 8 == 0 && x.xb < p.d)) && x.nch >= 1 && x.nch <= C::kChunks,
                      2);
    const uint32_t bytes = static_cast<uint32_t>(x.nch * p.R * 128 * (BWD ? 2 : 1));
    ptx::mbar_arrive_expect_tx(bar_full(st), bytes);
    const uint32_t sa = stage_addr(st);
    // general pe tiles read all d channels; every other tile reads through
    // tm_in0 / tm_in1 (clipped at channel nope under the general tiling)
    const CUtensorMap* m0 = (kGen && x.kind == 2) ? &p.tm_in0_pe : &p.tm_in0;
    for (int k = 0; k < x.nch; ++k) ptx::tma_load_2d(sa + k * kChunkBytes, m0, box_x(x, k), x.row0, bar_full(st));
    if (BWD) {
      const CUtensorMap* m1 = (kGen && x.kind == 2) ? &p.tm_in1_pe : &p.tm_in1;
      for (int k = 0; k < x.nch; ++k)
        ptx::tma_load_2d(sa + C::kTensorTile + k * kChunkBytes, m1, box_x(x, k), x.row0, bar_full(st));
    }
  };

  const int64_t G = gridDim.x;
  // forward: unused; backward: this CTA's static share of the first n_static tiles
  const int64_t t_begin = p.n_static * blockIdx.x / G;
  const int64_t t_end = p.n_static * (blockIdx.x + 1) / G;
  // The first tile needs no work counter (forward: tile blockIdx.x; backward:
  // the static share's first), so thread 0 loads it as soon as the barriers
  // exist, ahead of the rest of the set-up.
  const int64_t t_first = BWD ? t_begin : static_cast<int64_t>(blockIdx.x);
  const bool early = BWD ? t_begin < t_end : t_first < p.n_tiles;

  // M's bulk copy lands in the output ring (forward: and the buffers after it,
  // up to the rotation tables; backward: the ring alone, as X_lo behind it is
  // zeroed meanwhile). A copy that would not fit is not made, whatever the
  // host asked: the A build then reads M from L2.
  const bool m_copy = p.m_bulk != 0 &&
                      p.nh * p.gs * 4 <= (BWD ? C::kOutBufs * kChunkBytes : C::kOffTabEpi - C::kOffOut);

  // ------------------------------------------------------------ setup
  bool sched_mine = false;
  // forward launches with more than two tiles per CTA, backward ones with tail blocks
  const bool use_sched = p.sched != nullptr;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(bar_full(s), 1);
      ptx::mbar_init(bar_empty(s), 1);
    }
    for (int b = 0; b < OB; ++b) {
      ptx::mbar_init(bar_ob_full(b), 128);
      ptx::mbar_init(bar_ob_empty(b), 1);
    }
    for (int a = 0; a < NA; ++a) {
      ptx::mbar_init(bar_acc_full(a), BWD ? 1 : 2);
      ptx::mbar_init(bar_acc_empty(a), 128);
    }
    ptx::mbar_init(bar_x_full, 128);
    ptx::mbar_init(bar_x_empty, 1);
    ptx::mbar_init(bar_d2, 1);
    ptx::mbar_init(bar_done, 1);
    ptx::mbar_init(bar_x_go, 1);
    ptx::mbar_init(bar_m, 1);
    if constexpr (BWD) {
      for (int k = 0; k < 4; ++k) {
        ptx::mbar_init(bar_seg_full(k), 1);
        ptx::mbar_init(bar_seg_empty(k), 4);  // MMA thread, epilogue, store warp, transform warps
      }
      for (int b = 0; b < C::kNumD2; ++b) {
        if (b) ptx::mbar_init(bar_d2f(b), 1);
        ptx::mbar_init(bar_d2e(b), 128);
      }
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
    // M goes out first, ahead of every tile load (into the output ring, idle
    // until the first tile is mixed); the A build waits on it
    if (m_copy) {
      const uint32_t mbytes = static_cast<uint32_t>(p.nh * p.gs * 4);
      ptx::mbar_arrive_expect_tx(bar_m, mbytes);
      ptx::bulk_load(base + C::kOffOut, p.M, mbytes, bar_m);
    }
    if (early) {
      if (!BWD) stage_tile[0] = static_cast<int>(t_first);  // published by the load's barrier
      load_tile(0, t_first);
    }
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&p.tm_in0);
    ptx::prefetch_tmap(&p.tm_out);
    if (BWD) ptx::prefetch_tmap(&p.tm_in1);
  }
  if (warp == 1) {
    ptx::tmem_alloc(base + C::kOffMisc, C::kTmemCols);
    ptx::tmem_relinquish();
    // M into L2 ahead of the A build (128-byte lines); the warp reconverges
    // before anything warp-collective follows
    const char* mb = reinterpret_cast<const char*>(p.M);
    const int mbytes = p.nh * p.gs * 4;
    if (!m_copy)
      for (int o = lane * 128; o < mbytes; o += 32 * 128) ptx::prefetch_l2(mb + o);
    __syncwarp();
  }
  // Rows >= R of every 64-channel box are never loaded and must read as 0
  // (the MMA's K range covers them).
  if (p.R < kRowsMax) {
    const uint32_t tail = static_cast<uint32_t>(kRowsMax - p.R) * 128u;  // bytes per box
    const uint32_t nbox = static_cast<uint32_t>(S * C::kStageBytes / kChunkBytes);
    for (uint32_t o = threadIdx.x * 16u; o < nbox * tail; o += blockDim.x * 16u)
      ptx::st_shared_v4(base + C::kOffStage + (o / tail) * kChunkBytes + p.R * 128u + (o % tail), 0u, 0u, 0u, 0u);
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncwarp();  // thread 0 ran the set-up alone: its warp meets the barrier converged
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Backward segments, in the order every role runs them: segment 0 is the
  // static share (dM partial slot blockIdx.x), then the tail blocks this CTA
  // claimed (slot G + b). The producer publishes them through a 4-entry ring.
  auto tail_block = [&](uint32_t b, int64_t& t0, int64_t& t1) {
    const uint32_t na = static_cast<uint32_t>(p.tail_na), nab = na + static_cast<uint32_t>(p.tail_nb);
    const int64_t a_end = p.n_static + static_cast<int64_t>(na) * p.tail_ba;
    const int64_t b_end = a_end + static_cast<int64_t>(p.tail_nb) * p.tail_bb;
    if (b < na) {
      t0 = p.n_static + static_cast<int64_t>(b) * p.tail_ba;
      t1 = t0 + p.tail_ba;
    } else if (b < nab) {
      t0 = a_end + static_cast<int64_t>(b - na) * p.tail_bb;
      t1 = t0 + p.tail_bb;
    } else {
      t0 = b_end + static_cast<int64_t>(b - nab) * p.tail_bc;
      t1 = t0 + p.tail_bc;
    }
    if (t1 > p.n_tiles) t1 = p.n_tiles;
  };
  auto seg_publish = [&](uint32_t k, int64_t t0, int64_t t1, int slot) -> bool {
    const int e = static_cast<int>(k & 3u);
    if (!wait_bar(bar_seg_empty(e), ((k >> 2) & 1u) ^ 1u, abort_flag, (kRoleProducer << 8) | kBarSeg))
      return false;
    seg_ring[4 * e] = static_cast<int>(t0);
    seg_ring[4 * e + 1] = static_cast<int>(t1);
    seg_ring[4 * e + 2] = slot;
    ptx::mbar_arrive(bar_seg_full(e));  // release: the entry is visible to whoever sees the phase
    return true;
  };
  // one consumer thread reads segment k (t0 < 0: no more segments)
  auto seg_read = [&](uint32_t k, int64_t& t0, int64_t& t1, int& slot, unsigned code) -> bool {
    const int e = static_cast<int>(k & 3u);
    if (!wait_bar(bar_seg_full(e), (k >> 2) & 1u, abort_flag, code)) return false;
    t0 = seg_ring[4 * e];
    t1 = seg_ring[4 * e + 1];
    slot = seg_ring[4 * e + 2];
    ptx::mbar_arrive(bar_seg_empty(e));
    return true;
  };
  // a 128-thread group: its leader reads, the group learns it through bc[k & 1]
  auto seg_read_group = [&](uint32_t k, int64_t& t0, int64_t& t1, int& slot, unsigned code, bool leader,
                            volatile int* bc, uint32_t bar_id) -> bool {
    volatile int* b = bc + 4 * (k & 1u);
    if (leader) {
      int64_t a0 = 0, a1 = 0;
      int sl = 0;
      const bool ok = seg_read(k, a0, a1, sl, code);
      b[0] = ok ? 1 : 0;
      b[1] = static_cast<int>(a0);
      b[2] = static_cast<int>(a1);
      b[3] = sl;
    }
    ptx::named_bar_sync(bar_id, 128);
    if (!b[0]) return false;
    t0 = b[1];
    t1 = b[2];
    slot = b[3];
    return true;
  };

  // The producer starts streaming right away; meanwhile every other warp
  // builds A in TMEM and (backward) clears X_lo, then they meet at named
  // barrier 4 (all warps but the producer).
  if (warp != 0) {
    const int nthr = static_cast<int>(blockDim.x) - 32, tid = static_cast<int>(threadIdx.x) - 32;
    // the rotation frequencies (epilogue and transform warps read them after barrier 4)
    if (tid < half && tid < kMaxHalf) F[tid] = p.F[tid];
    if (warp >= 2 && warp < 6) {
      // A in TMEM: lane m holds row m; column kACol + hl*64 + j/2 holds the bf16
      // pair (j, j+1) of the hi (hl = 0) or lo (hl = 1) term, lower j in the
      // low half. Each thread reads its row's entries of M straight from L2,
      // all loads of a 64-column half in flight together.
      const uint32_t quad = static_cast<uint32_t>(warp & 3);
      const int m = static_cast<int>(quad * 32) + lane;
      const uint32_t row_addr = tmem_base + ((quad * 32u) << 16) + C::kACol;
      // Ungrouped M with a 16-byte-aligned start: M in shared memory once its
      // bulk copy has landed (the copy left ahead of every tile load);
      // otherwise the entries come from L2.
      const bool msm = m_copy;
      if (msm) wait_bar(bar_m, 0, abort_flag, (kRoleEpilogue << 8) | kBarM);
      const float* Msm = reinterpret_cast<const float*>(gbase + C::kOffOut);  // [nh][nh]
      if constexpr (STK) {
        // stacked A: lane m < 64 holds M^T_hi row m, lane 64 + h holds M^T_lo row h
        const MixLine col(p, m & 63, false);
        float v[64];
#pragma unroll
        for (int q = 0; q < 64; ++q) v[q] = msm ? Msm[q * 64 + (m & 63)] : col.at(q);
        uint32_t w[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const uint32_t hw = ptx::pack_bf16x2(v[2 * q], v[2 * q + 1]);
          w[q] = m < 64 ? hw : ptx::pack_bf16x2(v[2 * q] - ptx::bf16_lo_f32(hw), v[2 * q + 1] - ptx::bf16_hi_f32(hw));
        }
        ptx::tmem_st_x32(row_addr, w);
      } else {
        // A = blockdiag_P(M) (forward) or blockdiag_P(M^T) (backward): row m
        // (position m / nh, head m % nh) is nonzero on columns [pb, pb + nh) only
        const bool live = m < p.R;
        const int pb = live ? (m / p.nh) * p.nh : 0;
        const MixLine line(p, m - pb, !BWD);  // forward: row of M; backward: column
        // the 64-column half holding the block of the warp's first row goes
        // first, so that (nh = 64) every thread's loads go out in the first
        // round; the order must be the same across the warp (tcgen05.st is
        // warp-collective with one column address)
        const int m0 = static_cast<int>(quad * 32);
        const int kfirst = (m0 < p.R ? ((m0 / p.nh) * p.nh) >> 6 : 0) & 1;
        for (int i = 0; i < 2; ++i) {
          const int kh = i ^ kfirst;
          float v[64];
          if (msm && (p.nh & 63) != 0) {
            // M[g][o] (forward) or M[o][f] (backward) from shared memory
#pragma unroll
            for (int q = 0; q < 64; ++q) {
              const unsigned o = static_cast<unsigned>(kh * 64 + q - pb);
              v[q] = (live && o < static_cast<unsigned>(p.nh))
                         ? Msm[BWD ? static_cast<int>(o) * p.nh + (m - pb) : (m - pb) * p.nh + static_cast<int>(o)]
                         : 0.f;
            }
          } else if (msm && !BWD) {
            // nh % 64 == 0: this half lies wholly inside or outside the block
            const int o0 = kh * 64 - pb;  // first column of this half within the block
            if (live && o0 >= 0 && o0 < p.nh) {
              const float4* src =
                  reinterpret_cast<const float4*>(gbase + C::kOffOut) + ((m - pb) * p.nh + o0) / 4;
#pragma unroll
              for (int u = 0; u < 16; ++u) {
                const float4 t = src[u];
                v[4 * u] = t.x;
                v[4 * u + 1] = t.y;
                v[4 * u + 2] = t.z;
                v[4 * u + 3] = t.w;
              }
            } else {
#pragma unroll
              for (int q = 0; q < 64; ++q) v[q] = 0.f;
            }
          } else {
#pragma unroll
            for (int q = 0; q < 64; ++q) {
              const unsigned o = static_cast<unsigned>(kh * 64 + q - pb);
              v[q] = (live && o < static_cast<unsigned>(p.nh))
                         ? (msm ? Msm[static_cast<int>(o) * p.nh + (m - pb)] : line.at(static_cast<int>(o)))
                         : 0.f;
            }
          }
          uint32_t whi[32], wlo[32];
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            whi[q] = ptx::pack_bf16x2(v[2 * q], v[2 * q + 1]);
            wlo[q] = ptx::pack_bf16x2(v[2 * q] - ptx::bf16_lo_f32(whi[q]), v[2 * q + 1] - ptx::bf16_hi_f32(whi[q]));
          }
          ptx::tmem_st_x32(row_addr + kh * 32, whi);
          ptx::tmem_st_x32(row_addr + 64 + kh * 32, wlo);
        }
      }
      ptx::tmem_st_wait();
    }
    // X_lo starts at 0 on its nope channels
    if (BWD)
      for (uint32_t o = static_cast<uint32_t>(tid) * 16u; o < static_cast<uint32_t>(kChunkBytes);
           o += static_cast<uint32_t>(nthr) * 16u)
        ptx::st_shared_v4(base + C::kOffXlo + o, 0u, 0u, 0u, 0u);
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    ptx::named_bar_sync(4, nthr);
    ptx::tc_fence_after();
  }

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      // forward: the first two tiles are static (blockIdx.x, G + blockIdx.x),
      // later ones are claimed from the launch's counter, one claim ahead. Backward: the static share,
      // then tail blocks claimed one segment ahead, each segment published to
      // the other roles before its first tile is loaded.
      // The next tail block is claimed a few tiles before the current segment
      // ends, so that the claims come in the order in which CTAs run out of
      // work (the claim's latency hides behind those tiles' loads).
      constexpr int64_t kClaimAhead = 3;
      // Take the launch's counter slot (off the set-up's path: only the claims
      // need it). If another launch still holds it, claim nothing from it and
      // wind down (outputs undefined, fault recorded) once the first tile's
      // copies have landed.
      if (use_sched) sched_mine = sched_acquire(p.sched, launch_tag());
      if (use_sched && !sched_mine) {
        if (early) wait_bar_noabort(bar_full(0), 0);
        record_fault(BWD ? INVROPE_FAULT_SCHED_BUSY_BWD : INVROPE_FAULT_SCHED_BUSY_FWD, abort_flag);
      }
      // stage 0 holds the first tile; the forward's second is static too
      // (tile G + blockIdx.x), later ones come from the counter (2G + claim)
      int64_t t_next = early ? t_first + (BWD ? 1 : G) : t_first;
      int64_t seg_end = t_end;
      uint32_t seg_k = 0;
      uint32_t claim = 0xffffffffu;
      bool claimed = false;
      bool run = !*abort_flag;
      if constexpr (BWD) run = run && seg_publish(0, t_begin, t_end, static_cast<int>(blockIdx.x));
      for (uint32_t i = early ? 1u : 0u; run; ++i) {
        const int st = static_cast<int>(i % S);
        const uint32_t ph = (i / S) & 1u;
        if constexpr (BWD) {
          if (!claimed && p.n_tail > 0 && seg_end - t_next <= kClaimAhead) {
            claim = atomicAdd(&p.sched->next, 1u);
            claimed = true;
          }
          if (t_next >= seg_end) {
            ++seg_k;
            if (!claimed || claim >= static_cast<uint32_t>(p.n_tail)) {
              seg_publish(seg_k, -1, -1, -1);
              break;
            }
            int64_t a0 = 0, a1 = 0;
            tail_block(claim, a0, a1);
            if (!seg_publish(seg_k, a0, a1, static_cast<int>(G + claim))) break;
            t_next = a0;
            seg_end = a1;
            claimed = false;
            if (seg_end - t_next <= kClaimAhead) {
              claim = atomicAdd(&p.sched->next, 1u);
              claimed = true;
            }
          }
        }
        if (*abort_flag) break;
        if (!wait_bar(bar_empty(st), ph ^ 1u, abort_flag, (kRoleProducer << 8) | kBarEmpty)) break;
        const int64_t t = t_next;
        if (BWD) {
          t_next = t + 1;
        } else {
          if (t >= p.n_tiles) {
            stage_tile[st] = -1;  // published by the arrive below
            ptx::mbar_arrive(bar_full(st));
            break;
          }
          t_next = use_sched ? 2 * G + static_cast<int64_t>(atomicAdd(&p.sched->next, 1u)) : p.n_tiles;
          stage_tile[st] = static_cast<int>(t);
        }
        load_tile(st, t);
      }
      // every claim of this CTA is made: count it done on the slot now (the
      // launch's last CTA to do so frees it), off the kernel's final path
      if (use_sched && sched_mine) sched_release(p.sched, gridDim.x);
    }
    __syncwarp();  // the whole warp reaches the teardown barrier together
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t nks = static_cast<uint32_t>((p.R + 15) / 16);
      uint32_t d2_started = 0;  // bit b: D2 buffer b has taken a dM MMA in its segment
      int npe = 0;
      // A segment's first dM MMA into D2 buffer d2_wait_b waits until the drain
      // has read out the segment that used the buffer before (phase d2_par).
      int d2_wait_b = -1;
      uint32_t d2_par = 0;
      int cur_b = 0;   // D2 buffer of the segment being issued
      int owe_b = -1;  // STK: buffer whose segment is complete once the pending pe tile's chain is out
      // D2[b] += dY_tile * X_tile^T (both K-major, K = channels), plus dY_pe * X_lo^T on a pe tile.
      // STK: one M = 64 MMA per position into the same 64 x 64 accumulator
      // (row m in TMEM lane 32 (m / 16) + m % 16), rows 64p.. of both operands
      // 8 KB apart, so D2 holds the position sum itself.
      auto dm_chain = [&](int st, const Tile& x, int b) -> bool {
        if (b == d2_wait_b) {
          if (!wait_bar(bar_d2e(b), d2_par, abort_flag, (kRoleMma << 8) | kBarD2Empty)) return false;
          ptx::tc_fence_after();
          d2_wait_b = -1;
        }
        const uint32_t sa = stage_addr(st);
        const uint32_t d2 = tmem_base + C::kD2Col + static_cast<uint32_t>(b) * C::kD2Cols;
        uint32_t started = (d2_started >> b) & 1u;
        const uint32_t xa = sa + C::kTensorTile;
        if constexpr (STK) {
          const uint32_t idesc_dm = ptx::idesc_bf16_f32(64, 64, false, false);
          for (uint32_t ps = 0; ps < 2; ++ps)
            for (uint32_t kk = 0; kk < 4; ++kk) {
              const uint64_t ad = ptx::smem_desc_sw128(sa + ps * 8192u + kk * 32, 16, 1024);
              const uint64_t bd = ptx::smem_desc_sw128(xa + ps * 8192u + kk * 32, 16, 1024);
              ptx::tc_mma_ss(d2, ad, bd, idesc_dm, started);
              started = 1;
            }
          d2_started |= 1u << b;
          if (x.has_pe)
            for (uint32_t ps = 0; ps < 2; ++ps)
              for (uint32_t kk = 0; kk < 4; ++kk) {
                const uint64_t ad = ptx::smem_desc_sw128(sa + ps * 8192u + kk * 32, 16, 1024);
                const uint64_t bd = ptx::smem_desc_sw128(base + C::kOffXlo + ps * 8192u + kk * 32, 16, 1024);
                ptx::tc_mma_ss(d2, ad, bd, idesc_dm, 1);
              }
          return true;
        }
        const uint32_t idesc_dm = ptx::idesc_bf16_f32(128, 128, false, false);
        for (int k = 0; k < x.nch; ++k)
          for (uint32_t kk = 0; kk < 4; ++kk) {
            const uint64_t ad = ptx::smem_desc_sw128(sa + k * kChunkBytes + kk * 32, 16, 1024);
            const uint64_t bd = ptx::smem_desc_sw128(xa + k * kChunkBytes + kk * 32, 16, 1024);
            ptx::tc_mma_ss(d2, ad, bd, idesc_dm, started);
            started = 1;
          }
        d2_started |= 1u << b;
        if (x.has_pe) {
          // the lo terms of X: one box (the pe box of a regular tile) or both
          // boxes of a general pair block, X_lo box b pairing with dY box kpe + b
          const bool gen_pe = kGen && x.kind == 2;
          const int kpe = gen_pe ? 0 : (p.nope - x.c0) / kChunkCols;
          const int nlo = gen_pe ? 2 : 1;
          for (int b = 0; b < nlo; ++b)
            for (uint32_t kk = 0; kk < 4; ++kk) {
              const uint64_t ad = ptx::smem_desc_sw128(sa + (kpe + b) * kChunkBytes + kk * 32, 16, 1024);
              const uint64_t bd = ptx::smem_desc_sw128(base + C::kOffXlo + b * kChunkBytes + kk * 32, 16, 1024);
              ptx::tc_mma_ss(d2, ad, bd, idesc_dm, 1);
            }
        }
        return true;
      };
      // the pe tile whose dM chain is still to be issued (stage, tile, D2 buffer)
      int pend_st = -1, pend_b = 0;
      Tile pend_x{};
      auto flush_pending = [&]() {
        if (!wait_bar(bar_x_full, static_cast<uint32_t>(npe & 1), abort_flag, (kRoleMma << 8) | kBarXFull))
          return false;
        ptx::tc_fence_after();
        if (!dm_chain(pend_st, pend_x, pend_b)) return false;
        ptx::tc_commit(bar_empty(pend_st));
        ptx::tc_commit(bar_x_empty);
        ++npe;
        pend_st = -1;
        if (STK && owe_b >= 0) {  // that tile ended its segment: D2[owe_b] goes to the drain
          ptx::tc_commit(bar_d2f(owe_b));
          owe_b = -1;
        }
        return true;
      };
      // Backward: an outer loop over the segments, the per-tile loop within
      // a segment; the segment changes stay out of the per-tile loop, which is
      // the MMA thread's hot code. Forward: one pass of the per-tile loop.
      uint32_t seg_k = 0, i = 0;
      for (;;) {
        int64_t s_t = 0, s_t1 = 0;
        if constexpr (BWD) {
          int s_slot = 0;
          if (!seg_read(seg_k, s_t, s_t1, s_slot, (kRoleMma << 8) | kBarSeg)) break;
          ++seg_k;
          if (s_t < 0) break;
          // segment k = seg_k - 1 accumulates into D2 buffer k mod kNumD2,
          // after the drain of segment k - kNumD2 that used it before
          const uint32_t k = seg_k - 1;
          cur_b = STK ? static_cast<int>(k & 1u) : 0;
          d2_started &= ~(1u << cur_b);
          if (k >= static_cast<uint32_t>(C::kNumD2)) {
            d2_wait_b = cur_b;
            d2_par = ((k / C::kNumD2) - 1u) & 1u;
          }
        }
        bool seg_done = false;
      for (;; ++i) {
        const int st = static_cast<int>(i % S);
        const uint32_t ph = (i / S) & 1u;
        const int acc = acc_of(i);
        const uint32_t aph = acc_phase(i);
        int64_t t = 0;
        if constexpr (BWD) {
          if (s_t >= s_t1) {
            seg_done = true;
            break;
          }
          t = s_t++;
        }
        // Backward but the stacked kernel: the previous pe tile's dM chain goes
        // out as soon as its X is formed, before this tile's data is waited
        // for, so that its stage is free again while this one loads (issued
        // after this tile's head mix instead, it held its stage until this
        // tile had landed, and with two stages that left one load in flight:
        // nh = 128 535 -> 507 us, [65536, 16, 64 + 64] 203 -> 150 us). The
        // stacked kernel keeps the later place (4 stages; 134 vs 142 us at
        // [16384, 64, 0 + 64], 484 vs 486 us at the production shard). The
        // order is fixed either way, so dM stays reproducible.
        if (BWD && !STK && pend_st >= 0 && !flush_pending()) break;
        if (!wait_bar(bar_full(st), ph, abort_flag, (kRoleMma << 8) | kBarFull)) break;
        if (!BWD) t = static_cast<int64_t>(stage_tile[st]);
        if (!BWD && t < 0) {
          // pass the end of the tile stream on to the epilogue
          if (!wait_bar(bar_acc_empty(acc), aph ^ 1u, abort_flag, (kRoleMma << 8) | kBarAccEmpty)) break;
          acc_tile[acc] = -1;
          ptx::mbar_arrive(bar_acc_full(acc));
          ptx::tc_commit(bar_acc_full(acc));
          break;
        }
        const Tile x = decode_tile<BWD, WIDE, GEN>(p, t);
        INVROPE_DBG_CHECK(st < S && acc < NA && t >= 0 && t < p.n_tiles, 3);
        // The transform warps only see pe tiles; this thread has observed every
        // stage phase in order, so it tells them when the pe tile has landed.
        // They take one hand-off at a time: when every tile is a pe tile (one
        // channel tile) the previous one is still pending here, and this tile
        // is handed over only after that one's flush below (its X used), so two
        // hand-offs never complete on bar_x_go before they have seen the first.
        const bool handoff_early = BWD && x.has_pe && pend_st < 0;
        if (handoff_early) ptx::mbar_arrive(bar_x_go);
        if (!wait_bar(bar_acc_empty(acc), aph ^ 1u, abort_flag, (kRoleMma << 8) | kBarAccEmpty)) break;
        ptx::tc_fence_after();
        const uint32_t sa = stage_addr(st);
        // head mix: D[acc] = A_hi * B + A_lo * B, A in TMEM, B = the tile (MN-major, K = rows)
        const uint32_t d_acc = tmem_base + static_cast<uint32_t>(acc) * acc_cols;
        if constexpr (STK) {
          // stacked: D[128 x 128] = [M^T_hi ; M^T_lo] * [tile rows 0-63 | tile rows 64-127],
          // K = the 64 heads of a position (A in TMEM); N block 1 sits 64 rows
          // (8 KB) below N block 0
          const uint32_t idesc_stk = ptx::idesc_bf16_f32(128, 128, false, true);
          for (uint32_t ks = 0; ks < 4; ++ks) {
            const uint64_t bd = ptx::smem_desc_sw128(sa + ks * 2048, 64 * 128, 1024);
            ptx::tc_mma_ts(d_acc, tmem_base + C::kACol + ks * 8, bd, idesc_stk, ks != 0);
          }
        } else {
          const uint32_t idesc_mix = ptx::idesc_bf16_f32(128, 64u * x.nch, false, true);
          for (uint32_t hl = 0; hl < 2; ++hl)
            for (uint32_t ks = 0; ks < nks; ++ks) {
              const uint64_t bd = ptx::smem_desc_sw128(sa + ks * 2048, kChunkBytes, 1024);
              ptx::tc_mma_ts(d_acc, tmem_base + C::kACol + hl * 64 + ks * 8, bd, idesc_mix, (hl | ks) != 0);
            }
        }
        if (!BWD) acc_tile[acc] = static_cast<int>(t);
        ptx::tc_commit(bar_acc_full(acc));  // the epilogue may start once the mix is done
        if (!BWD) {
          ptx::mbar_arrive(bar_acc_full(acc));  // publishes acc_tile[acc]
          ptx::tc_commit(bar_empty(st));        // the input stage is free once the mix is done
          continue;
        }
        // dM share. A pe tile's chain needs the transform warps' X, so it is
        // issued one tile late, after the next tile's MMAs: the tensor pipe and
        // the input ring keep moving while X is formed. The issue order is fixed
        // by the tile sequence alone, so D2 (and dM) stay reproducible.
        if (!x.has_pe) {
          if (!dm_chain(st, x, cur_b)) break;
          ptx::tc_commit(bar_empty(st));
        }
        if (pend_st >= 0 && !flush_pending()) break;
        if (x.has_pe && !handoff_early) ptx::mbar_arrive(bar_x_go);
        if (x.has_pe) {
          pend_st = st;
          pend_b = cur_b;
          pend_x = x;
        }
      }
        if (!seg_done) break;  // forward: the end of the tile stream; else a wait gave up
        // The segment is issued. D2 goes to the drain (transform warps) once
        // every MMA so far completes, after the segment's last dM chain: with
        // one D2 buffer the pending pe tile's chain goes out now; with two it
        // keeps its usual place one tile later (in the next segment) and the
        // hand-over follows it.
        if constexpr (STK) {
          if (pend_st >= 0)
            owe_b = cur_b;
          else
            ptx::tc_commit(bar_d2f(cur_b));
        } else {
          if (pend_st >= 0 && !flush_pending()) break;
          ptx::tc_commit(bar_d2);
        }
      }
      if constexpr (STK) {
        if (pend_st >= 0) flush_pending();  // the last segment ended with a pe tile
      }
      // every MMA issued must complete before TMEM is freed, abort or not
      ptx::tc_commit(bar_done);
      wait_bar_noabort(bar_done, 0);
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
    uint32_t n = 0;  // output chunk counter (output ring position)
    bool ok = true;
    // backward: the next tile's (row tile, channel tile), advanced without a
    // division within a segment [s_t, s_t1); the segments in an outer loop
    int e_rt = 0, e_ct = 0;
    uint32_t seg_k = 0, i = 0;
    for (;;) {
      int64_t s_t = 0, s_t1 = 0;
      if constexpr (BWD) {
        int sl = 0;
        if (!seg_read_group(seg_k, s_t, s_t1, sl, (kRoleEpilogue << 8) | kBarSeg, e == 0, seg_bc_epi, 1)) break;
        ++seg_k;
        if (s_t < 0) break;
        const Tile x0 = decode_tile<BWD, WIDE, GEN>(p, s_t);
        e_rt = x0.rt;
        e_ct = x0.ct;
      }
      bool seg_done = false;
    for (; ok; ++i) {
      int64_t t = 0;
      if constexpr (BWD) {
        if (s_t >= s_t1) {
          seg_done = true;
          break;
        }
        t = s_t++;
      }
      const int acc = acc_of(i);
      const uint32_t aph = acc_phase(i);
      if (stk) {
        // one group barrier for both waits: this tile's accumulator and its output buffer
        volatile int* slot = slot_epi + (i & 1);
        if (e == 0) {
          const int b = static_cast<int>(n % OB);
          *slot = wait_bar(bar_acc_full(acc), aph, abort_flag, (kRoleEpilogue << 8) | kBarAccFull) &&
                          wait_bar(bar_ob_empty(b), ((n / OB) & 1u) ^ 1u, abort_flag,
                                   (kRoleEpilogue << 8) | kBarOut)
                      ? 1
                      : 0;
        }
        ptx::named_bar_sync(1, 128);
        if (*slot == 0) break;
      } else if (!group_wait(bar_acc_full(acc), aph, abort_flag, (kRoleEpilogue << 8) | kBarAccFull, e == 0,
                             slot_epi + (i & 1), 1)) {
        break;
      }
      ptx::tc_fence_after();
      if (!BWD) t = static_cast<int64_t>(acc_tile[acc]);
      if (!BWD && t < 0) {
        // pass the end of the tile stream on to the store warp
        const int b = static_cast<int>(n % OB);
        if (group_wait(bar_ob_empty(b), ((n / OB) & 1u) ^ 1u, abort_flag,
                       (kRoleEpilogue << 8) | kBarOut, e == 0, slot_ob + (n & 1), 1)) {
          if (e == 0) ob_tile[b] = -1;
          ptx::mbar_arrive(bar_ob_full(b));
        }
        break;
      }
      const Tile x = BWD ? make_tile<BWD, WIDE, GEN>(p, e_rt, e_ct) : decode_tile<BWD, WIDE, GEN>(p, t);
      if (BWD && ++e_ct == p.n_ct) {
        e_ct = 0;
        ++e_rt;
      }
      if (kGen && x.kind == 2) {
        // General pair block: accumulator columns [0, 64) are box 0, [64, 128)
        // box 1; pair ii has its first half at column da + ii and its second
        // half at column db + ii. Rotate, round once, store both halves
        // straight to global memory (the boxes also hold channels of other
        // pairs, so they are not stored whole).
        fill_rot_table_gen(tab, F, p, x.s0, x.j, x.np, e, 128);
        ptx::named_bar_sync(1, 128);
        const uint32_t ta = tmem_base + lane_addr + static_cast<uint32_t>(acc) * acc_cols;
        const int c1 = p.nope + 32 * x.j, c2 = c1 + half;
        const int da = c1 - x.xa, db = kChunkCols + c2 - x.xb;
        const int64_t grow = static_cast<int64_t>(x.row0) + r;
        const bool live = row_ok && grow < p.rows;
        uint16_t* yrow = p.out + grow * p.d;
        const float2* rt = tab + pl * 32;
        if (x.j == 0)  // nope channels [xa, nope): plain head mix, rounded once
          for (int ii = 0; ii < da; ++ii) {
            uint32_t a;
            ptx::tmem_ld_x1(ta + ii, a);
            ptx::tmem_ld_wait(a);
            if (live) yrow[x.xa + ii] = bf16_bits(__uint_as_float(a));
          }
        if (da == 0 && db == kChunkCols && (x.np & 7) == 0) {
          for (int i0 = 0; i0 < x.np; i0 += 8) {
            uint32_t a[8], bb[8];
            ptx::tmem_ld_x8(ta + i0, a);
            ptx::tmem_ld_x8(ta + kChunkCols + i0, bb);
            ptx::tmem_ld_wait(a, bb);
            if (live) {
              uint32_t w1[4], w2[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                float y1[2], y2[2];
#pragma unroll
                for (int s2 = 0; s2 < 2; ++s2) {
                  const int kq = 2 * q + s2;
                  const float2 cs = rt[i0 + kq];
                  const float x1 = __uint_as_float(a[kq]), x2 = __uint_as_float(bb[kq]);
                  y1[s2] = x1 * cs.x - sgn * x2 * cs.y;
                  y2[s2] = x2 * cs.x + sgn * x1 * cs.y;
                }
                w1[q] = ptx::pack_bf16x2(y1[0], y1[1]);
                w2[q] = ptx::pack_bf16x2(y2[0], y2[1]);
              }
              *reinterpret_cast<uint4*>(yrow + c1 + i0) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
              *reinterpret_cast<uint4*>(yrow + c2 + i0) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
            }
          }
        } else {
          for (int ii = 0; ii < x.np; ++ii) {
            uint32_t a, bb;
            ptx::tmem_ld_x1(ta + da + ii, a);
            ptx::tmem_ld_x1(ta + db + ii, bb);
            ptx::tmem_ld_wait(a, bb);
            if (live) {
              const float2 cs = rt[ii];
              const float x1 = __uint_as_float(a), x2 = __uint_as_float(bb);
              yrow[c1 + ii] = bf16_bits(x1 * cs.x - sgn * x2 * cs.y);
              yrow[c2 + ii] = bf16_bits(x2 * cs.x + sgn * x1 * cs.y);
            }
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_acc_empty(acc));
        continue;
      }
      const int pcol = p.nope - x.c0;  // tile-relative column of the first pe channel
      if (x.has_pe) {
        fill_rot_table(tab, F, p, x.s0, half, e, 128);
        ptx::named_bar_sync(1, 128);
      }
      const uint32_t taddr = tmem_base + lane_addr + static_cast<uint32_t>(acc) * acc_cols;
      INVROPE_DBG_CHECK((static_cast<uint32_t>(acc) + 1u) * acc_cols <= static_cast<uint32_t>(C::kD2Col), 4);
      for (int k = 0; k < x.nch; ++k, ++n) {
        const int b = static_cast<int>(n % OB);
        if (!stk && !group_wait(bar_ob_empty(b), ((n / OB) & 1u) ^ 1u, abort_flag,
                                (kRoleEpilogue << 8) | kBarOut, e == 0, slot_ob + (n & 1), 1)) {
          ok = false;
          break;
        }
        const uint32_t ob = out_addr(b);
        const bool pe_chunk = x.has_pe && (pcol >> 6) == k;
        const bool pe_whole = pe_chunk && half == 32;  // the pe block is exactly this chunk
        if (stk) {
          // Stacked mix: lane h < 64 (quads 0, 1) holds the hi rows of head h,
          // lane 64 + h (quads 2, 3) its lo rows; D column 64 p + c is channel c
          // of position p, whose output row is 64 p + h. Each warp pair splits
          // the work by position: the hi warps finish position 0 and hand their
          // position-1 terms (fp32, exchange rows) to the lo warps, which finish
          // position 1 and hand over their position-0 terms through the output
          // buffer as bf16 (a lo term is ~2^-9 of the result, so that rounding
          // costs ~2^-17 relative).
          const int h = r & 63;
          const bool hi = quad < 2;
          const uint32_t xrow = base + C::kOffXch + static_cast<uint32_t>(h) * 256u;
          const uint32_t hx = static_cast<uint32_t>(h & 7);  // unit c of a row sits at (c ^ hx) * 16
          // both halves out of TMEM in one round trip; the accumulator is then free
          uint32_t v[64], y[64];  // y: this warp's own position (hi: 0, lo: 1)
          ptx::tmem_ld_x64(taddr + (hi ? 64 : 0), v);
          ptx::tmem_ld_x64(taddr + (hi ? 0 : 64), y);
          ptx::tmem_ld_wait(v, y);
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar_acc_empty(acc));
          {
            if (hi) {
#pragma unroll
              for (int c = 0; c < 16; ++c)
                ptx::st_shared_v4(xrow + ((static_cast<uint32_t>(c) ^ hx) << 4), v[4 * c], v[4 * c + 1],
                                  v[4 * c + 2], v[4 * c + 3]);
            } else {
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const uint32_t* w = v + 8 * u;
                ptx::st_shared_v4(swz_unit_addr(ob, h, 8 * u),
                                  ptx::pack_bf16x2(__uint_as_float(w[0]), __uint_as_float(w[1])),
                                  ptx::pack_bf16x2(__uint_as_float(w[2]), __uint_as_float(w[3])),
                                  ptx::pack_bf16x2(__uint_as_float(w[4]), __uint_as_float(w[5])),
                                  ptx::pack_bf16x2(__uint_as_float(w[6]), __uint_as_float(w[7])));
              }
            }
          }
          ptx::named_bar_sync(3, 128);  // both halves are parked
          const int pp = hi ? 0 : 1;
          const int row = pp * 64 + h;
          if (hi) {
            uint32_t l[32];
#pragma unroll
            for (int u = 0; u < 8; ++u)
              ptx::ld_shared_v4(swz_unit_addr(ob, h, 8 * u), l[4 * u], l[4 * u + 1], l[4 * u + 2], l[4 * u + 3]);
#pragma unroll
            for (int q = 0; q < 32; ++q) {
              y[2 * q] = __float_as_uint(__uint_as_float(y[2 * q]) + ptx::bf16_lo_f32(l[q]));
              y[2 * q + 1] = __float_as_uint(__uint_as_float(y[2 * q + 1]) + ptx::bf16_hi_f32(l[q]));
            }
          } else {
            uint32_t f[64];
#pragma unroll
            for (int c = 0; c < 16; ++c)
              ptx::ld_shared_v4(xrow + ((static_cast<uint32_t>(c) ^ hx) << 4), f[4 * c], f[4 * c + 1],
                                f[4 * c + 2], f[4 * c + 3]);
#pragma unroll
            for (int k = 0; k < 64; ++k) y[k] = __float_as_uint(__uint_as_float(y[k]) + __uint_as_float(f[k]));
          }
          if (pe_chunk) {
            // the chunk is the whole pe block: pairs (i, 32 + i)
            const float2* rt = tab + pp * 32;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float2 cs = rt[i];
              const float x1 = __uint_as_float(y[i]), x2 = __uint_as_float(y[32 + i]);
              y[i] = __float_as_uint(x1 * cs.x - sgn * x2 * cs.y);
              y[32 + i] = __float_as_uint(x2 * cs.x + sgn * x1 * cs.y);
            }
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint32_t* w = y + 8 * u;
            ptx::st_shared_v4(swz_unit_addr(ob, row, 8 * u),
                              ptx::pack_bf16x2(__uint_as_float(w[0]), __uint_as_float(w[1])),
                              ptx::pack_bf16x2(__uint_as_float(w[2]), __uint_as_float(w[3])),
                              ptx::pack_bf16x2(__uint_as_float(w[4]), __uint_as_float(w[5])),
                              ptx::pack_bf16x2(__uint_as_float(w[6]), __uint_as_float(w[7])));
          }
        } else {
          if (!pe_whole) {
            // one 64-column TMEM load, one wait, then 8 swizzled 16-byte stores
            uint32_t v[64];
            ptx::tmem_ld_x64(taddr + k * kChunkCols, v);
            ptx::tmem_ld_wait(v);
            if (row_ok) {
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const uint32_t w0 = ptx::pack_bf16x2(__uint_as_float(v[8 * u + 0]), __uint_as_float(v[8 * u + 1]));
                const uint32_t w1 = ptx::pack_bf16x2(__uint_as_float(v[8 * u + 2]), __uint_as_float(v[8 * u + 3]));
                const uint32_t w2 = ptx::pack_bf16x2(__uint_as_float(v[8 * u + 4]), __uint_as_float(v[8 * u + 5]));
                const uint32_t w3 = ptx::pack_bf16x2(__uint_as_float(v[8 * u + 6]), __uint_as_float(v[8 * u + 7]));
                ptx::st_shared_v4(swz_unit_addr(ob, r, 8 * u), w0, w1, w2, w3);
              }
            }
          }
          if (pe_whole) {
            // pe = 64 filling the chunk: one load brings both halves of every pair
            const float2* rt = tab + pl * 32;
            uint32_t v[64];
            ptx::tmem_ld_x64(taddr + pcol, v);
            ptx::tmem_ld_wait(v);
            if (row_ok) {
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                uint32_t w1[4], w2[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  float y1[2], y2[2];
#pragma unroll
                  for (int s2 = 0; s2 < 2; ++s2) {
                    const int kq = 8 * u + 2 * q + s2;
                    const float2 cs = rt[kq];
                    const float x1 = __uint_as_float(v[kq]), x2 = __uint_as_float(v[32 + kq]);
                    y1[s2] = x1 * cs.x - sgn * x2 * cs.y;
                    y2[s2] = x2 * cs.x + sgn * x1 * cs.y;
                  }
                  w1[q] = ptx::pack_bf16x2(y1[0], y1[1]);
                  w2[q] = ptx::pack_bf16x2(y2[0], y2[1]);
                }
                ptx::st_shared_v4(swz_unit_addr(ob, r, 8 * u), w1[0], w1[1], w1[2], w1[3]);
                ptx::st_shared_v4(swz_unit_addr(ob, r, 32 + 8 * u), w2[0], w2[1], w2[2], w2[3]);
              }
            }
          } else if (pe_chunk) {
            // rotate the pe pairs of the fp32 accumulator, then round once
            const int qcol = pcol - k * kChunkCols;  // chunk-relative
            const float2* rt = tab + pl * half;
            if ((half & 7) == 0) {
              for (int i0 = 0; i0 < half; i0 += 8) {
                uint32_t a[8], bb[8];
                ptx::tmem_ld_x8(taddr + pcol + i0, a);
                ptx::tmem_ld_x8(taddr + pcol + half + i0, bb);
                ptx::tmem_ld_wait(a, bb);
                if (row_ok) {
                  uint32_t w1[4], w2[4];
#pragma unroll
                  for (int q = 0; q < 4; ++q) {
                    float y1[2], y2[2];
#pragma unroll
                    for (int s2 = 0; s2 < 2; ++s2) {
                      const int kq = 2 * q + s2;
                      const float2 cs = rt[i0 + kq];
                      const float x1 = __uint_as_float(a[kq]), x2 = __uint_as_float(bb[kq]);
                      y1[s2] = x1 * cs.x - sgn * x2 * cs.y;
                      y2[s2] = x2 * cs.x + sgn * x1 * cs.y;
                    }
                    w1[q] = ptx::pack_bf16x2(y1[0], y1[1]);
                    w2[q] = ptx::pack_bf16x2(y2[0], y2[1]);
                  }
                  ptx::st_shared_v4(swz_unit_addr(ob, r, qcol + i0), w1[0], w1[1], w1[2], w1[3]);
                  ptx::st_shared_v4(swz_unit_addr(ob, r, qcol + half + i0), w2[0], w2[1], w2[2], w2[3]);
                }
              }
            } else {
              for (int ii = 0; ii < half; ++ii) {
                uint32_t a, bb;
                ptx::tmem_ld_x1(taddr + pcol + ii, a);
                ptx::tmem_ld_x1(taddr + pcol + half + ii, bb);
                ptx::tmem_ld_wait(a, bb);
                if (row_ok) {
                  const float2 cs = rt[ii];
                  const float x1 = __uint_as_float(a), x2 = __uint_as_float(bb);
                  const int c1 = qcol + ii, c2 = qcol + half + ii;
                  st_shared_b16(swz_unit_addr(ob, r, c1) + (c1 & 7) * 2, bf16_bits(x1 * cs.x - sgn * x2 * cs.y));
                  st_shared_b16(swz_unit_addr(ob, r, c2) + (c2 & 7) * 2, bf16_bits(x2 * cs.x + sgn * x1 * cs.y));
                }
              }
            }
          }
        }
        // hand the finished 64-channel chunk to the store warp
        if (!BWD && e == 0) {
          ob_tile[b] = static_cast<int>(t);
          ob_chunk[b] = k;
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(bar_ob_full(b));
      }
      if (!stk) {  // the stacked path releases its accumulator right after its TMEM loads
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_acc_empty(acc));
      }
    }
      if (!seg_done) break;
    }
  } else if (warp == C::kWarpStore) {
    // ---------------------------------------------------------- TMA store (output ring)
    if (lane == 0) {
      constexpr int kIn = C::kOutInflight;
      uint32_t n = 0;
      bool ok = true;
      uint32_t seg_k = 0;
      for (;;) {
        int64_t s_t = 0, s_t1 = 0;
        if constexpr (BWD) {
          int sl = 0;
          if (!seg_read(seg_k, s_t, s_t1, sl, (kRoleStore << 8) | kBarSeg)) break;
          ++seg_k;
          if (s_t < 0) break;
        }
        bool seg_done = false;
      for (; ok;) {
        int64_t tb = 0;
        if constexpr (BWD) {
          if (s_t >= s_t1) {
            seg_done = true;
            break;
          }
          tb = s_t++;
        }
        // forward: one chunk per hand-off; backward: every box of a tile, none
        // of a general pair block (stored directly by the epilogue)
        int nk = 1;
        if (BWD) {
          const Tile xb = decode_tile<BWD, WIDE, GEN>(p, tb);
          nk = (kGen && xb.kind == 2) ? 0 : xb.nch;
        }
        for (int kk = 0; kk < nk; ++kk, ++n) {
          const int b = static_cast<int>(n % OB);
          if (!wait_bar(bar_ob_full(b), (n / OB) & 1u, abort_flag,
                        (kRoleStore << 8) | kBarOut)) {
            ok = false;
            break;
          }
          const int64_t t = BWD ? tb : static_cast<int64_t>(ob_tile[b]);
          if (!BWD && t < 0) {
            ok = false;
            break;
          }
          const int k = BWD ? kk : ob_chunk[b];
          const Tile x = decode_tile<BWD, WIDE, GEN>(p, t);
          INVROPE_DBG_CHECK(b < OB && k < x.nch && x.kind != 2 && box_x(x, k) < p.d, 6);
          ptx::tma_store_2d(&p.tm_out, out_addr(b), box_x(x, k), x.row0);
          ptx::bulk_commit();
          // keep kIn stores reading; recycle the buffer of the oldest finished one
          if (n + 1u >= static_cast<uint32_t>(kIn)) {
            ptx::bulk_wait_read<kIn - 1>();
            ptx::mbar_arrive(bar_ob_empty(static_cast<int>((n - (kIn - 1)) % OB)));
          }
        }
      }
        if (!seg_done) break;
      }
      ptx::bulk_wait<0>();
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- X = invrope(O) on the pe chunk (bwd)
    if constexpr (BWD) {
      const int xr = threadIdx.x - 192;
      float2* tab = reinterpret_cast<float2*>(gbase + C::kOffTabXf);
      int npe = 0;
      uint32_t i = 0;
      // D2 of segment k -> dM partial slot `slot`: the diagonal nh x nh blocks
      // of D2 (one per position of a tile), summed over positions. Row r of D2
      // (position pl = r / nh, head g) holds its block's row in columns
      // [pl nh, pl nh + nh). The D2 columns are handed back (bar_d2_empty) as
      // soon as they are read.
      auto drain_d2 = [&](uint32_t k, int slot) -> bool {
        // segment k used D2 buffer k mod kNumD2
        const int b = static_cast<int>(k % C::kNumD2);
        if (!group_wait(bar_d2f(b), (k / C::kNumD2) & 1u, abort_flag, (kRoleTransform << 8) | kBarD2, xr == 0,
                        slot_d2, 2))
          return false;
        ptx::tc_fence_after();
        const uint32_t q4 = static_cast<uint32_t>(warp & 3);
        const int r = static_cast<int>(q4 * 32u) + lane;  // this thread's TMEM lane: D2 row r
        const uint32_t taddr = tmem_base + ((q4 * 32u) << 16) + C::kD2Col + static_cast<uint32_t>(b) * C::kD2Cols;
        const bool rok = r < p.R;
        const int nh = p.nh;
        const int pl = rok ? r / nh : 0, g = r - pl * nh;
        const int lo = pl * nh, hi = lo + nh;
        float* dst = p.ws + static_cast<int64_t>(slot) * nh * nh;
        if constexpr (STK) {
          // D2 is the position-summed 64 x 64 block: row g in lane 32 (g / 16) +
          // g % 16, so lanes 0-15 of each warp hold rows 16 q4 .. 16 q4 + 15.
          // The other D2 buffer takes the next segment meanwhile, so nothing
          // waits for this hand-back.
          uint32_t v[64];
          ptx::tmem_ld_x64(taddr, v);
          ptx::tmem_ld_wait(v);
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar_d2e(b));
          if (lane < 16) {
            float4* drow = reinterpret_cast<float4*>(dst + static_cast<int64_t>(q4 * 16u + lane) * 64);
#pragma unroll
            for (int u = 0; u < 16; ++u)
              drow[u] = make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                    __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
          }
        } else if (p.P == 1) {
          // one position per tile: D2 row r is partial row r
          for (int j0 = 0; j0 < nh; j0 += 32) {
            uint32_t v[32];
            ptx::tmem_ld_x32(taddr + j0, v);
            ptx::tmem_ld_wait(v);
            if (!rok) continue;
            float* drow = dst + static_cast<int64_t>(r) * nh;
            if (j0 + 32 <= nh && (nh & 3) == 0) {
#pragma unroll
              for (int u = 0; u < 8; ++u)
                *reinterpret_cast<float4*>(drow + j0 + 4 * u) =
                    make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
            } else {
#pragma unroll
              for (int jj = 0; jj < 32; ++jj)
                if (j0 + jj < nh) drow[j0 + jj] = __uint_as_float(v[jj]);
            }
          }
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar_d2e(b));
        } else if (p.P == 2) {
          // Position 1's rows park theirs in X_lo (free now: the segment's last
          // dM chain has completed), row g at g * 64 with column c at c ^ (g & 31)
          // (conflict-free); position 0's rows add them and write the partial.
          float* xch = reinterpret_cast<float*>(gbase + C::kOffXlo);
          for (int j0 = 0; j0 < 128; j0 += 32) {
            if (!__any_sync(0xffffffffu, rok && pl == 1 && j0 < hi && j0 + 32 > lo)) continue;
            uint32_t v[32];
            ptx::tmem_ld_x32(taddr + j0, v);
            ptx::tmem_ld_wait(v);
            if (rok && pl == 1) {
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) {
                const int j = j0 + jj;
                if (j >= lo && j < hi) xch[g * 64 + ((j - lo) ^ (g & 31))] = __uint_as_float(v[jj]);
              }
            }
          }
          ptx::named_bar_sync(2, 128);
          for (int j0 = 0; j0 < 128; j0 += 32) {
            if (!__any_sync(0xffffffffu, rok && pl == 0 && j0 < nh)) continue;
            uint32_t v[32];
            ptx::tmem_ld_x32(taddr + j0, v);
            ptx::tmem_ld_wait(v);
            if (rok && pl == 0) {
              float* drow = dst + static_cast<int64_t>(g) * nh;
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) {
                const int j = j0 + jj;
                if (j < nh) drow[j] = __uint_as_float(v[jj]) + xch[g * 64 + (j ^ (g & 31))];
              }
            }
          }
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar_d2e(b));
          ptx::named_bar_sync(2, 128);  // every row has read X_lo
          // X_lo back to zero: the pe transform writes only its pe columns
          for (uint32_t o = static_cast<uint32_t>(xr) * 16u; o < static_cast<uint32_t>(C::kXloBytes); o += 128u * 16u)
            ptx::st_shared_v4(base + C::kOffXlo + o, 0u, 0u, 0u, 0u);
          ptx::fence_proxy_async_smem();
        } else {
          // P > 2 positions per tile: such launches have one segment (no tail),
          // so this runs after the CTA's last MMA and the input ring is free.
          // red[h * (R + 1) + r] = D2[r][pl nh + h] (odd row stride: the
          // transposed reads below are conflict-free), then position sums.
          float* red = reinterpret_cast<float*>(gbase + C::kOffStage);
          const int rs = p.R + 1;
          for (int j0 = 0; j0 < 128; j0 += 32) {
            uint32_t v[32];
            ptx::tmem_ld_x32(taddr + j0, v);
            ptx::tmem_ld_wait(v);
            if (rok) {
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) {
                const int j = j0 + jj;
                if (j >= lo && j < hi) red[(j - lo) * rs + r] = __uint_as_float(v[jj]);
              }
            }
          }
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar_d2e(b));
          ptx::named_bar_sync(2, 128);
          const int nn = nh * nh;
          // consecutive threads take consecutive h: coalesced partial rows
          for (int idx = xr; idx < nn; idx += 128) {
            const int gg = idx / nh, h = idx - gg * nh;
            float sum = 0.f;
            for (int q = 0; q < p.P; ++q) sum += red[h * rs + q * nh + gg];
            dst[idx] = sum;
          }
        }
        return true;
      };
      uint32_t seg_k = 0;
      for (;;) {
        int64_t s_t0 = 0, s_t1 = 0;
        int s_slot = 0;
        if (!seg_read_group(seg_k, s_t0, s_t1, s_slot, (kRoleTransform << 8) | kBarSeg, xr == 0, seg_bc_xf, 2))
          break;
        if (s_t0 < 0) break;
        int64_t t = s_t0;
      for (; t < s_t1; ++t, ++i) {
        const Tile x = decode_tile<BWD, WIDE, GEN>(p, t);
        if (!x.has_pe) continue;
        const int st = static_cast<int>(i % S);
        const uint32_t ph = (i / S) & 1u;
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
        if (kGen && x.kind == 2) {
          // General pair block: X = invrope(O) for its pairs (first halves in
          // O box 0 at column da + ii, second halves in box 1 at db + ii), hi
          // in place, lo into X_lo; every other column of both boxes is set to
          // 0 in both, so that dM counts each channel once (in its own tile).
          fill_rot_table_gen(tab, F, p, x.s0, x.j, x.np, xr, 128);
          ptx::named_bar_sync(2, 128);
          if (xr < p.R) {
            const uint32_t oc = stage_addr(st) + C::kTensorTile;
            const uint32_t xl = base + C::kOffXlo;
            const int c1 = p.nope + 32 * x.j, c2 = c1 + half;
            const int da = c1 - x.xa, db = kChunkCols + c2 - x.xb;
            const int np = x.np;
            const float2* rt = tab + (xr / p.nh) * 32;
            if (da == 0 && db == kChunkCols && (np & 7) == 0) {
              for (int i0 = 0; i0 < np; i0 += 8) {
                const uint32_t a1 = swz_unit_addr(oc, xr, i0);
                const uint32_t a2 = swz_unit_addr(oc, xr, kChunkCols + i0);
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
                ptx::st_shared_v4(swz_unit_addr(xl, xr, i0), l1[0], l1[1], l1[2], l1[3]);
                ptx::st_shared_v4(swz_unit_addr(xl, xr, kChunkCols + i0), l2[0], l2[1], l2[2], l2[3]);
              }
              for (int u = np >> 3; u < 8; ++u)
                for (int bx = 0; bx < 2; ++bx) {
                  ptx::st_shared_v4(swz_unit_addr(oc, xr, bx * kChunkCols + 8 * u), 0u, 0u, 0u, 0u);
                  ptx::st_shared_v4(swz_unit_addr(xl, xr, bx * kChunkCols + 8 * u), 0u, 0u, 0u, 0u);
                }
            } else {
              for (int ii = 0; ii < np; ++ii) {
                const int k1 = da + ii, k2 = db + ii;
                const uint32_t a1 = swz_unit_addr(oc, xr, k1) + (k1 & 7) * 2;
                const uint32_t a2 = swz_unit_addr(oc, xr, k2) + (k2 & 7) * 2;
                const float x1 = bf16_bits_to_f32(ld_shared_b16(a1));
                const float x2 = bf16_bits_to_f32(ld_shared_b16(a2));
                const float2 cs = rt[ii];
                const float X1 = x1 * cs.x + x2 * cs.y, X2 = x2 * cs.x - x1 * cs.y;
                const uint16_t hb1 = bf16_bits(X1), hb2 = bf16_bits(X2);
                st_shared_b16(a1, hb1);
                st_shared_b16(a2, hb2);
                st_shared_b16(swz_unit_addr(xl, xr, k1) + (k1 & 7) * 2, bf16_bits(X1 - bf16_bits_to_f32(hb1)));
                st_shared_b16(swz_unit_addr(xl, xr, k2) + (k2 & 7) * 2, bf16_bits(X2 - bf16_bits_to_f32(hb2)));
              }
              // pair block 0 owns the nope channels [xa, nope) in columns
              // [0, da): X = O there (hi as loaded, lo 0)
              const int own0 = x.j == 0 ? da : 0;
              for (int k = 0; k < 2 * kChunkCols; ++k) {
                if ((k >= da && k < da + np) || (k >= db && k < db + np)) continue;
                if (k >= own0) st_shared_b16(swz_unit_addr(oc, xr, k) + (k & 7) * 2, 0);
                st_shared_b16(swz_unit_addr(xl, xr, k) + (k & 7) * 2, 0);
              }
            }
          }
          ptx::fence_proxy_async_smem();
          ptx::mbar_arrive(bar_x_full);
          ++npe;
          continue;
        }
        fill_rot_table(tab, F, p, x.s0, half, xr, 128);
        ptx::named_bar_sync(2, 128);
        if (xr < p.R) {
          const int kpe = (p.nope - x.c0) / kChunkCols;
          INVROPE_DBG_CHECK(kpe >= 0 && kpe < x.nch && st < S, 5);
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
        if (t < s_t1) break;  // a wait gave up: the CTA is winding down
        if (!drain_d2(seg_k, s_slot)) break;
        ++seg_k;
      }
    }
  }

  // ------------------------------------------------------------ teardown
  // M's bulk copy must have landed before the CTA leaves (it has, unless the
  // CTA gave up early): bounded wait that ignores the abort flag
  if (m_copy && threadIdx.x == 0) wait_bar_noabort(bar_m, 0);
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// dM[o] = sum of the CTA partials ws[c][src(o)] (each [nh, nh]) in a fixed
// order. A thread block takes 32 outputs (one per lane); warp w sums partials
// c = w, w + 32, ... in fp32 with a compensation term (Kahan), and warp 0
// then adds the 32 warp sums in order. fp64 arithmetic is scarce on this GPU,
// so the per-element adds stay in fp32; the compensated sum keeps the error
// near one fp32 rounding of the total. A grouped mix keeps only the diagonal
// blocks: output o = (k, i, j) of [nh/gs, gs, gs] reads entry (k gs + i, k gs + j).
constexpr int kReduceWarps = 32;

__global__ void __launch_bounds__(32 * kReduceWarps)
    dm_reduce_kernel(const float* __restrict__ ws, float* __restrict__ dM, int nparts, int nh, int gs) {
  __shared__ float part_s[kReduceWarps][33];
  __shared__ float part_c[kReduceWarps][33];
  ptx::griddep_wait();  // launched early (programmatic dependent launch): wait for the partials
  const int nn = nh * nh, n_out = nh * gs;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int idx = blockIdx.x * 32 + tx;
  const int k = idx / (gs * gs), rem = idx - k * gs * gs;
  const int src = (k * gs + rem / gs) * nh + k * gs + rem % gs;
  float sum = 0.f, comp = 0.f;
  if (idx < n_out) {
#pragma unroll 8
    for (int c = ty; c < nparts; c += kReduceWarps) {
      const float y = __ldg(ws + static_cast<int64_t>(c) * nn + src) - comp;
      const float t = sum + y;
      comp = (t - sum) - y;
      sum = t;
    }
  }
  part_s[ty][tx] = sum;
  part_c[ty][tx] = comp;
  __syncthreads();
  if (ty == 0 && idx < n_out) {
    float s2 = 0.f, c2 = 0.f;
    for (int w = 0; w < kReduceWarps; ++w) {
      const float y = part_s[w][tx] - (part_c[w][tx] + c2);
      const float t = s2 + y;
      c2 = (t - s2) - y;
      s2 = t;
    }
    dM[idx] = s2;
  }
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

// Encoded tensor maps of recent calls: a map depends only on the pointer and
// the view's geometry, so a caller that reuses its buffers (every layer of a
// model does) skips the encoding. Small, round-robin, one lock.
struct TmapKey {
  const void* ptr;
  int64_t rows;
  int d, width, box_rows;
  bool operator==(const TmapKey& o) const {
    return ptr == o.ptr && rows == o.rows && d == o.d && width == o.width && box_rows == o.box_rows;
  }
};
struct TmapCache {
  static constexpr int kEntries = 32;
  std::mutex mu;
  TmapKey key[kEntries] = {};
  CUtensorMap map[kEntries];
  bool used[kEntries] = {};
  int next = 0;
};
TmapCache g_tmap_cache;

bool encode_tmap(CUtensorMap* m, const void* ptr, int64_t rows, int d, int width, int box_rows);

// 2-D bf16 view [rows, d] (row stride d) with 64 x box_rows boxes, 128-byte
// swizzle. Channels at or beyond `width` (<= d) lie outside the view: loads
// read them as zero and stores leave them alone.
bool make_tmap(CUtensorMap* m, const void* ptr, int64_t rows, int d, int width, int box_rows) {
  const TmapKey k{ptr, rows, d, width, box_rows};
  TmapCache& c = g_tmap_cache;
  {
    std::lock_guard<std::mutex> lock(c.mu);
    for (int i = 0; i < TmapCache::kEntries; ++i)
      if (c.used[i] && c.key[i] == k) {
        *m = c.map[i];
        return true;
      }
  }
  if (!encode_tmap(m, ptr, rows, d, width, box_rows)) return false;
  std::lock_guard<std::mutex> lock(c.mu);
  const int i = c.next;
  c.next = (c.next + 1) % TmapCache::kEntries;
  c.key[i] = k;
  c.map[i] = *m;
  c.used[i] = true;
  return true;
}

bool encode_tmap(CUtensorMap* m, const void* ptr, int64_t rows, int d, int width, int box_rows) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kChunkCols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rotary frequency f_i = theta^(-2i/pe) as turns per position in 0.64 fixed
// point: the kernel reduces pos * F[i] mod 2^64 exactly to a fractional turn.
// The last (pe, theta) table of each host thread is kept.
void fill_freq(uint64_t* F, int pe, double theta) {
  thread_local int last_pe = 0;
  thread_local double last_theta = 0.0;
  thread_local uint64_t last_F[kMaxHalf];
  const int n = pe / 2 < kMaxHalf ? pe / 2 : kMaxHalf;
  if (pe != last_pe || theta != last_theta) {
    for (int i = 0; i < n; ++i) {
      const double f = std::pow(theta, -2.0 * i / pe);
      last_F[i] = static_cast<uint64_t>(std::llround(std::ldexp(f * 0.15915494309189535, 63))) << 1;
    }
    last_pe = pe;
    last_theta = theta;
  }
  std::memcpy(F, last_F, sizeof(uint64_t) * n);
}

struct Shape {
  int P = 0, R = 0, n_ct = 0, n_nope_ct = 0;
  int64_t n_tiles = 0;
  bool gen = false;   // general tiling: the pe block does not lie inside one 64-channel box
  bool wide = false;  // backward: 128-channel tiles (one position per tile, or the general tiling)
  bool stacked = false;  // backward, nh = 64, pe block = one whole chunk: the stacked kernel
  bool tail_ok = false;  // backward: the kernel can hand out tail blocks (the stacked one)
};

// Validate a postmix shape and lay out its tiles (forward, or backward if bwd).
int check_shape(int64_t sq, int nh, int nope, int pe, bool bwd, Shape* s) {
  if (sq < 0 || nh < 1 || nope < 0 || pe < 2 || (pe & 1)) return INVROPE_ERR_INVALID_ARG;
  const int64_t d = static_cast<int64_t>(nope) + pe;
  if (d % 8 != 0 || d > (1 << 20)) return INVROPE_ERR_INVALID_ARG;
  if (nh > 128) return INVROPE_ERR_UNSUPPORTED;
  // rows of the [sq*nh, d] view are 32-bit TMA coordinates
  if (sq * nh >= (int64_t(1) << 31)) return INVROPE_ERR_UNSUPPORTED;
  s->gen = nope / kChunkCols != (d - 1) / kChunkCols;
  // backward: the stacked kernel for nh = 64 with the pe block on one whole
  // 64-channel chunk (the production shape), 128-channel tiles for every other
  // shape (measured 6-11% faster than 64-channel tiles at nh < 64 and for other
  // nh = 64 shapes: half the head-mix MMA instructions per byte), except tiny
  // ones without the general tiling (tensors under 1 MiB: there the 64-channel
  // kernel starts ~2 us sooner)
  s->stacked = bwd && nh == 64 && pe == kChunkCols && nope % kChunkCols == 0;
  s->wide = bwd && !s->stacked && (s->gen || sq * nh * d * 2 >= (int64_t(1) << 20));
  const int nc = (!bwd || s->wide) ? 2 * kChunkCols : kChunkCols;
  const int pmax = (bwd && s->gen) ? kPosPerTileMax : kPosPerTileMaxFwd;
  s->P = 128 / nh < pmax ? 128 / nh : pmax;
  s->R = s->P * nh;
  // tail blocks: the stacked kernel, whose double-buffered D2 makes segment
  // changes free (the 128-channel kernel's CTAs finish within ~25 us of each
  // other under the static split, and a single D2's hand-back costs more)
  s->tail_ok = s->stacked;
  if (!s->gen) {
    s->n_nope_ct = 0;
    s->n_ct = static_cast<int>((d + nc - 1) / nc);
  } else {
    s->n_nope_ct = ((nope & ~7) + nc - 1) / nc;
    s->n_ct = s->n_nope_ct + (pe / 2 + 31) / 32;
  }
  s->n_tiles = ((sq + s->P - 1) / s->P) * s->n_ct;
  if (s->n_tiles >= (int64_t(1) << 31)) return INVROPE_ERR_UNSUPPORTED;
  return INVROPE_OK;
}

// The tensor maps of a launch: in0 (and in1) read, out written. Under the
// general tiling the maps of the nope tiles end at channel nope & ~7, and the
// pair blocks read through the full-width *_pe maps.
bool make_maps(PostmixParams* p, const Shape& s, const void* in0, const void* in1, void* out, int64_t rows,
               int nope, int d) {
  // (a clip must fall on a 16-byte boundary: channels [nope & ~7, nope) go
  // with the first pair block)
  const int width = (s.gen && (nope & ~7) > 0) ? (nope & ~7) : d;
  if (!make_tmap(&p->tm_in0, in0, rows, d, width, s.R) || !make_tmap(&p->tm_out, out, rows, d, width, s.R))
    return false;
  if (in1 && !make_tmap(&p->tm_in1, in1, rows, d, width, s.R)) return false;
  if (!in1) p->tm_in1 = p->tm_in0;
  if (!s.gen) {
    p->tm_in0_pe = p->tm_in0;
    p->tm_in1_pe = p->tm_in1;
    return true;
  }
  if (!make_tmap(&p->tm_in0_pe, in0, rows, d, d, s.R)) return false;
  if (in1 && !make_tmap(&p->tm_in1_pe, in1, rows, d, d, s.R)) return false;
  if (!in1) p->tm_in1_pe = p->tm_in0_pe;
  return true;
}

template <bool BWD, bool WIDE = false, bool STK = false, bool GEN = true>
int ensure_smem_attr(int device) {
  static std::mutex mu;
  static bool done[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return INVROPE_ERR_DEVICE;
  if (!done[device]) {
    const cudaError_t err = cudaFuncSetAttribute(postmix_kernel<BWD, WIDE, STK, GEN>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 KCfg<BWD, WIDE, STK, (!BWD || WIDE) && GEN>::kSmemAlloc);
    if (err != cudaSuccess) return cuda_fail(err);
    done[device] = true;
  }
  return INVROPE_OK;
}

bool valid_theta(double theta) { return std::isfinite(theta) && theta > 0.0; }

SlotRing g_sched_ring;

}  // namespace

int reset_postmix_sched(int device) { return slot_reset_all(g_sched_ring, &g_sched, device); }

int occupy_postmix_slot(int device, unsigned long long owner) {
  SchedSlot* s = nullptr;
  const int st = slot_peek_eager(g_sched_ring, &g_sched, device, &s);
  if (st != INVROPE_OK) return st;
  const cudaError_t err = cudaMemcpy(&s->owner, &owner, sizeof(owner), cudaMemcpyHostToDevice);
  return err == cudaSuccess ? INVROPE_OK : cuda_fail(err);
}

// Grid size of the backward kernel.
static int64_t bwd_grid(const Shape& s, int sms) { return s.n_tiles < sms ? s.n_tiles : sms; }

// The backward's schedule: each CTA's static share of the first n_static
// tiles, then n_tail fixed tail blocks handed out one at a time, so that
// CTAs on SMs that draw more memory bandwidth take more of the tail (per-SM
// bandwidth differs by several percent). Every static share and every tail
// block has its own dM partial slot, so dM does not depend on which CTA ran
// what. A tail needs the drain's position sum to run mid-kernel (at most 2
// positions per tile) and enough tiles per CTA to be worth it; the partial
// slots stay within 8 MiB (or twice the static slots).
struct TailPlan {
  int64_t n_static = 0;
  int n_tail = 0, na = 0, ba = 0, nb = 0, bb = 0, bc = 0;
};

static TailPlan bwd_tail_plan(const Shape& s, int64_t grid, int nh) {
  TailPlan t;
  t.n_static = s.n_tiles;
  const int64_t per = s.n_tiles / (grid > 0 ? grid : 1);
  const int64_t slot_bytes = static_cast<int64_t>(nh) * nh * 4;
  if (s.P > 2 || per < 96) return t;
  if (!s.tail_ok) return t;
  const int64_t budget = std::max<int64_t>(int64_t(8) << 20, 2 * grid * slot_bytes);
  const int64_t max_tail = budget / slot_bytes - grid;
  if (max_tail < grid) return t;
  // Blocks shrink as the tail runs out (~11% of the tiles in all): half as
  // many as CTAs of ~1/11 of a share (the CTAs that finish their share
  // first), one per CTA of ~1/22, and the rest of the slots in blocks of
  // ~1/54 of a share for the end.
  t.ba = static_cast<int>(std::max<int64_t>(4, per / 11));
  t.bb = static_cast<int>(std::max<int64_t>(2, per / 22));
  t.bc = static_cast<int>(std::max<int64_t>(1, per / 54));
  t.na = static_cast<int>(grid / 2);
  t.nb = static_cast<int>(std::min<int64_t>(grid, max_tail - t.na));
  const int64_t nc = std::max<int64_t>(0, std::min<int64_t>(max_tail - t.na - t.nb, grid));
  const int64_t tail = static_cast<int64_t>(t.na) * t.ba + static_cast<int64_t>(t.nb) * t.bb + nc * t.bc;
  t.n_static = s.n_tiles - tail;
  t.n_tail = static_cast<int>(t.na + t.nb + nc);
  return t;
}

// Bytes of dM partials a backward launch writes: one [nh, nh] slot per CTA
// and per tail block.
static size_t bwd_partial_bytes(const Shape& s, int64_t grid, int nh) {
  const TailPlan t = bwd_tail_plan(s, grid, nh);
  return static_cast<size_t>(grid + t.n_tail) * nh * nh * sizeof(float);
}

}  // namespace invrope

using namespace invrope;

// Arguments shared by both directions beyond the shape: group size and the
// optional positions array (validated here; pointers checked by the callers).
static int check_mix_args(int nh, int gs, const int32_t* positions, int64_t pos0, double theta) {
  if (gs < 1 || gs > nh || nh % gs != 0) return INVROPE_ERR_INVALID_ARG;
  if (pos0 < 0 || !valid_theta(theta)) return INVROPE_ERR_INVALID_ARG;
  if (positions && !aligned(positions, 4)) return INVROPE_ERR_INVALID_ARG;
  return INVROPE_OK;
}

extern "C" int invrope_postmix_fwd_ex(const void* O, const float* M, void* Y, int64_t sq, int nh, int gs,
                                      int nope, int pe, const int32_t* positions, int64_t pos0, double theta,
                                      struct CUstream_st* stream) {
  Shape s;
  int st = check_shape(sq, nh, nope, pe, false, &s);
  if (st != INVROPE_OK) return st;
  if ((st = check_mix_args(nh, gs, positions, pos0, theta)) != INVROPE_OK) return st;
  if (sq == 0) return INVROPE_OK;
  if (!O || !M || !Y || !aligned(O, 16) || !aligned(Y, 16) || !aligned(M, 4)) return INVROPE_ERR_INVALID_ARG;
  const size_t tbytes = static_cast<size_t>(sq) * nh * (nope + pe) * 2;
  const size_t mbytes = static_cast<size_t>(nh) * gs * 4;
  const size_t pbytes = positions ? static_cast<size_t>(sq) * 4 : 0;
  if (overlaps(Y, tbytes, O, tbytes) || overlaps(Y, tbytes, M, mbytes) || overlaps(Y, tbytes, positions, pbytes))
    return INVROPE_ERR_INVALID_ARG;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != INVROPE_OK) return st;
  if ((st = ensure_smem_attr<false>(dev.device)) != INVROPE_OK) return st;
  PostmixParams p;
  std::memset(&p, 0, sizeof(p));
  const int d = nope + pe;
  if (!make_maps(&p, s, O, nullptr, Y, sq * nh, nope, d)) return INVROPE_ERR_CUDA;
  p.out = static_cast<uint16_t*>(Y);
  p.M = M;
  p.ws = nullptr;
  // The first two tiles of each CTA are static: a launch with no more tiles
  // than that claims nothing and needs no work-counter slot.
  const int64_t grid = s.n_tiles < dev.sms ? s.n_tiles : dev.sms;
  p.sched = nullptr;
  if (s.n_tiles > 2 * grid &&
      (st = slot_take(g_sched_ring, &g_sched, dev.device, reinterpret_cast<cudaStream_t>(stream), &p.sched)) !=
          INVROPE_OK)
    return st;
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
  p.pos = positions;
  p.gs = gs;
  p.gen = s.gen ? 1 : 0;
  p.n_nope_ct = s.n_nope_ct;
  p.rows = sq * nh;
  p.log2_theta = std::log2(theta);
  p.n_static = s.n_tiles;
  // M by one bulk copy at kernel start: 16-byte aligned, ungrouped, a whole
  // number of 16-byte units (nh even)
  p.m_bulk = (aligned(M, 16) && gs == nh && nh % 2 == 0) ? 1 : 0;
  fill_freq(p.F, pe, theta);
  postmix_kernel<false><<<static_cast<unsigned>(grid), KCfg<false>::kThreads, KCfg<false>::kSmemAlloc,
                          reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return check_launch();
}

extern "C" int invrope_postmix_fwd(const void* O, const float* M, void* Y, int64_t sq, int nh, int nope, int pe,
                                   int64_t pos0, double theta, struct CUstream_st* stream) {
  return invrope_postmix_fwd_ex(O, M, Y, sq, nh, nh, nope, pe, nullptr, pos0, theta, stream);
}

extern "C" size_t invrope_postmix_bwd_workspace_bytes(int64_t sq, int nh, int nope, int pe) {
  Shape s;
  if (check_shape(sq, nh, nope, pe, true, &s) != INVROPE_OK) return 0;
  DeviceInfo dev;
  if (current_device(&dev) != INVROPE_OK) return 0;
  if (sq == 0) return static_cast<size_t>(nh) * nh * sizeof(float);
  return bwd_partial_bytes(s, bwd_grid(s, dev.sms), nh);
}

extern "C" int invrope_postmix_bwd_ex(const void* dY, const void* O, const float* M, void* dO, float* dM,
                                      void* workspace, size_t workspace_bytes, int64_t sq, int nh, int gs,
                                      int nope, int pe, const int32_t* positions, int64_t pos0, double theta,
                                      struct CUstream_st* stream) {
  Shape s;
  int st = check_shape(sq, nh, nope, pe, true, &s);
  if (st != INVROPE_OK) return st;
  if ((st = check_mix_args(nh, gs, positions, pos0, theta)) != INVROPE_OK) return st;
  if (!M || !dM || !aligned(M, 4) || !aligned(dM, 4)) return INVROPE_ERR_INVALID_ARG;
  if (sq > 0 && (!dY || !O || !dO || !aligned(dY, 16) || !aligned(O, 16) || !aligned(dO, 16)))
    return INVROPE_ERR_INVALID_ARG;
  const size_t tbytes = static_cast<size_t>(sq) * nh * (nope + pe) * 2;
  const size_t mbytes = static_cast<size_t>(nh) * gs * 4;
  const size_t pbytes = positions ? static_cast<size_t>(sq) * 4 : 0;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != INVROPE_OK) return st;
  const int64_t grid = sq == 0 ? 0 : bwd_grid(s, dev.sms);
  const TailPlan tail = grid > 0 ? bwd_tail_plan(s, grid, nh) : TailPlan{};
  const size_t need = grid == 0 ? static_cast<size_t>(nh) * nh * sizeof(float) : bwd_partial_bytes(s, grid, nh);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return INVROPE_ERR_WORKSPACE;
  const void* outs[3] = {dO, dM, workspace};
  const size_t out_bytes[3] = {tbytes, mbytes, need};
  const void* ins[4] = {dY, O, M, positions};
  const size_t in_bytes[4] = {tbytes, tbytes, mbytes, pbytes};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 4; ++j)
      if (overlaps(outs[i], out_bytes[i], ins[j], in_bytes[j])) return INVROPE_ERR_INVALID_ARG;
    for (int j = i + 1; j < 3; ++j)
      if (overlaps(outs[i], out_bytes[i], outs[j], out_bytes[j])) return INVROPE_ERR_INVALID_ARG;
  }
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (grid > 0) {
    const bool wide = s.wide;
    // the 128-channel kernel comes in two builds: with the general tiling's
    // pair blocks, and without (its code made the nh = 128 backward ~13 us slower)
    if ((st = wide        ? (s.gen ? ensure_smem_attr<true, true, false, true>(dev.device)
                                   : ensure_smem_attr<true, true, false, false>(dev.device))
              : s.stacked ? ensure_smem_attr<true, false, true>(dev.device)
                          : ensure_smem_attr<true>(dev.device)) != INVROPE_OK)
      return st;
    PostmixParams p;
    std::memset(&p, 0, sizeof(p));
    const int d = nope + pe;
    if (!make_maps(&p, s, dY, O, dO, sq * nh, nope, d)) return INVROPE_ERR_CUDA;
    p.out = static_cast<uint16_t*>(dO);
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
    // stacked head mix: two positions of 64 heads per tile, pe block = one chunk
    p.stacked = s.stacked ? 1 : 0;
    p.pos = positions;
    p.gs = gs;
    p.gen = s.gen ? 1 : 0;
    p.n_nope_ct = s.n_nope_ct;
    p.rows = sq * nh;
    p.log2_theta = std::log2(theta);
    // M by one bulk copy at kernel start, as in the forward (it lands in the
    // output ring, idle until the first tile is mixed), when it fits there:
    // the X_lo buffer behind the ring is zeroed while the copy may still be
    // landing. Otherwise (nh = 128) the A build reads M from L2.
    // (the ring of the exact build launched below)
    const int out_ring = (wide        ? (s.gen ? KCfg<true, true, false, true>::kOutBufs
                                               : KCfg<true, true, false, false>::kOutBufs)
                          : s.stacked ? KCfg<true, false, true>::kOutBufs
                                      : KCfg<true>::kOutBufs) *
                         kChunkBytes;
    p.m_bulk = (aligned(M, 16) && gs == nh && nh % 2 == 0 && nh * gs * 4 <= out_ring) ? 1 : 0;
    p.n_static = tail.n_static;
    p.n_tail = tail.n_tail;
    p.tail_na = tail.na;
    p.tail_ba = tail.ba;
    p.tail_nb = tail.nb;
    p.tail_bb = tail.bb;
    p.tail_bc = tail.bc;
    p.sched = nullptr;
    if (tail.n_tail > 0 &&
        (st = slot_take(g_sched_ring, &g_sched, dev.device, cs, &p.sched)) != INVROPE_OK)
      return st;
    fill_freq(p.F, pe, theta);
    if (wide && s.gen)
      postmix_kernel<true, true, false, true>
          <<<static_cast<unsigned>(grid), KCfg<true, true>::kThreads, KCfg<true, true>::kSmemAlloc, cs>>>(p);
    else if (wide)
      postmix_kernel<true, true, false, false><<<static_cast<unsigned>(grid), KCfg<true, true, false, false>::kThreads,
                                                 KCfg<true, true, false, false>::kSmemAlloc, cs>>>(p);
    else if (s.stacked)
      postmix_kernel<true, false, true><<<static_cast<unsigned>(grid), KCfg<true, false, true>::kThreads,
                                          KCfg<true, false, true>::kSmemAlloc, cs>>>(p);
    else  // tiny shapes: 64-channel tiles
      postmix_kernel<true><<<static_cast<unsigned>(grid), KCfg<true>::kThreads, KCfg<true>::kSmemAlloc, cs>>>(p);
    if ((st = check_launch()) != INVROPE_OK) return st;
  }
  // Programmatic dependent launch: the reduction grid's launch is processed
  // while the main kernel drains, and its blocks wait in-kernel (griddepcontrol)
  // for the main kernel's partials. The main kernel does not signal early:
  // reduction blocks that start early crowd onto the first SMs to free up.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((nh * gs + 31) / 32));
  cfg.blockDim = dim3(32 * kReduceWarps);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = cs;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = grid > 0 ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, dm_reduce_kernel, static_cast<const float*>(workspace), dM,
                                             static_cast<int>(grid + tail.n_tail), nh, gs);
  if (err != cudaSuccess) return cuda_fail(err);
  return check_launch();
}

extern "C" int invrope_postmix_bwd(const void* dY, const void* O, const float* M, void* dO, float* dM,
                                   void* workspace, size_t workspace_bytes, int64_t sq, int nh, int nope, int pe,
                                   int64_t pos0, double theta, struct CUstream_st* stream) {
  return invrope_postmix_bwd_ex(dY, O, M, dO, dM, workspace, workspace_bytes, sq, nh, nh, nope, pe, nullptr, pos0,
                                theta, stream);
}

extern "C" int invrope_watchdog_selftest(int64_t limit_us, int* fault) {
  if (!fault || limit_us < 1000 || limit_us > 2000000) return INVROPE_ERR_INVALID_ARG;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != INVROPE_OK) return st;
  int stale = 0;
  if ((st = invrope_take_device_fault(&stale)) != INVROPE_OK) return st;  // start from a clear flag
  watchdog_selftest_kernel<<<1, 32>>>(static_cast<uint64_t>(limit_us) * 1000u);
  if ((st = check_launch()) != INVROPE_OK) return st;
  return invrope_take_device_fault(fault);
}

extern "C" int invrope_take_device_fault(int* fault) {
  if (!fault) return INVROPE_ERR_INVALID_ARG;
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return cuda_fail(err);
  if ((err = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(err);
  unsigned v = 0, vr = 0;
  if ((err = cudaMemcpyFromSymbol(&v, g_fault_code, sizeof(v))) != cudaSuccess) return cuda_fail(err);
  const unsigned zero = 0;
  if ((err = cudaMemcpyToSymbol(g_fault_code, &zero, sizeof(zero))) != cudaSuccess) return cuda_fail(err);
  int st = take_remap_fault(&vr);
  if (st != INVROPE_OK) return st;
  if (v == 0) v = vr;
  // After a fault a launch may have left a work-counter slot held (its
  // blocks that found the slot busy never release it): nothing runs on the
  // device now, so every slot is returned to the free state.
  if (v != 0 && ((st = reset_postmix_sched(device)) != INVROPE_OK || (st = reset_remap_sched(device)) != INVROPE_OK))
    return st;
  *fault = static_cast<int>(v);
  return INVROPE_OK;
}
