// svdq_kernel.cuh -- persistent, warp-specialised sm_103a kernel for
//
//     y = scaled_mma(act4, wgt4) * wcscale + bias + lora_act_in @ lora_up
//
// ("SVDQuant W4A4 on Blackwell" §2 operator, §3.1 NVFP4 block-scaled MMA with
// scales in tensor memory, §3.2 CTA pair sharing one MMA, §3.5 static
// persistent tile scheduler, §3.6 / §6 warp specialisation, §6.3 LoRA
// accumulated into the same tensor-memory accumulator, §6.6 fused per-column
// affine epilogue).
//
// Template parameters: CG = CTAs per MMA (1, or 2 for a CTA pair issuing
// cta_group::2 MMAs of M = 256), BN = output columns per tile, KBI = K blocks
// per ring item (1), F16 = fp16 instead of bf16 16-bit I/O, SK = split-K
// instance.  Each CTA owns 128 output rows; in a pair the leader (cluster
// rank 0) issues every MMA, A is split along M and B along N between the two
// CTAs' shared memory.
//
// Row-quad order.  Inside every 128-row block of an operand tile, tile row
// a + 32b (a < 32, b < 4) holds matrix row 4a + b.  The TMA builds this order
// itself from a 3-D view of the row-major operand (dims: bytes, row quads,
// row within the quad).  A and B tiles, the LoRA rows and the output store all
// use it, so the product is unchanged; what it buys is the scale layout: the
// tensor-memory word of lane a, column b must hold the four group scales of
// tile row a + 32b = matrix row 4a + b, and those are four consecutive bytes
// of each raw [group][row] scale row.  One 32-bit shared load per group and a
// 4x4 byte transpose in registers give a lane its words: no staging, no
// exchange between warps.  In tensor memory the accumulator's lanes follow the
// row order (warp q's lane a is output row 4a + q) and its columns the B order
// (column 128h + a + 32b is output column 128h + 4a + b).
//
// 19 warps per CTA (608 threads):
//   warps 0, 12, 13  TMA producers, one thread each, every ring item split
//                three ways (one issuing thread streams far fewer bytes per
//                second than three): warp 0 the [16 groups x rows] scale
//                boxes, the LoRA item rows and the leader's byte count; warp 12
//                the packed act tiles; warp 13 the packed wgt tiles (128-byte
//                swizzle).  LoRA ring item (32 ranks): raw fp32 LA rows, 16-bit
//                LU rows (64-byte swizzle) and wcscale.
//   warps 1, 14  MMA issuers (one thread each, leader CTA), alternating ring
//                items and taking turns (a turn barrier per issuer keeps the
//                items in ring order): tcgen05.mma kind::mxf4nvf4
//                block_scale.scale_vec::4X for main items, kind::f16 (bf16 or
//                fp16) for LoRA items, commits that free ring stages / publish
//                accumulators.
//   warps 2, 3   LoRA operand builders: LU' = round16(LU / wc), a quarter of
//                the rows each (the scale feeders take the other half), in place
//                in the stage's K-major swizzled layout (nothing to do for
//                prepacked weights, whose LU' arrives ready).
//   warps 4..7, 15..18  epilogue, two warps per 32-lane quadrant, each taking
//                half of the tile's 32-column groups: tcgen05.ld -> fma(acc,
//                wc, bias) -> 16-bit -> shared staging (64-byte swizzle) -> one
//                TMA tile store per group; every column read is cleared for the
//                next tile and each warp releases the accumulator after its
//                last group (the MMA waits for all eight).
//   warps 8..11  scale feeders: turn the stage's scale boxes into row-per-lane
//                words in registers (a 4x4 byte transpose of raw scales, or
//                plain 16-byte loads of scale words: prepacked weights,
//                activation scales handed over packed) and write
//                them into tensor memory with tcgen05.st (one warp per 32-lane
//                quadrant), off the MMA pipe; on LoRA items they build
//                LA' = round16(LA), 32 rows each, and scale their share of LU'.
// The MMA issuers, the LoRA builders and the scale feeders run a unit's LoRA
// items and its K-block items in two loops, the feeders' K-block loop once per
// scale layout: a per-item branch on the item kind or the layout cost 6-20 %
// through the register allocation of the loop.
// Warp w accesses tensor-memory lanes 32(w%4) .. 32(w%4)+31, so epilogue warps
// 4..7 and 15..18 and scale feeders 8..11 each cover all four quadrants.
//
// Per unit of work (an output tile, or with split-K one of its K ranges) the
// ring carries ceil(R/32) LoRA items (on the first split only), then its main
// items; every role walks the same item sequence, so stage index and phase
// bit survive unit boundaries.  Split-K units that are not a tile's last split
// store an fp32 partial tile and raise a per-launch flag; the last split adds
// them in tensor memory before its epilogue.  Every MMA accumulates into an
// accumulator the epilogue has cleared, so no LoRA or block-scaled MMA waits
// for another to complete; the two issuers take turns, so items reach the
// tensor core in ring order and results are bit-reproducible.  LU' is pre-divided
// by wcscale, so the epilogue's acc * wcscale restores LA @ LU unscaled, as the
// operator states.
//
// Every mbarrier wait is bounded by %globaltimer; on expiry the kernel records
// SVDQ_ERR_TIMEOUT and the wait site, every role leaves its loop, in-flight
// tcgen05 work is drained with a second bounded wait, in-flight TMA loads get
// a fixed grace period, tensor memory is freed and the CTA exits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"

namespace svdq {

constexpr int kThreads = 608;
constexpr int kBM = 128;     // output rows per CTA (per-CTA MMA M)
constexpr int kBK = 256;     // K elements per K block (128 packed bytes per row)
constexpr int kLoraRanks = 32;  // ranks per LoRA ring item
constexpr int kMaxStages = 8;
constexpr int kTmemCols = 512;
constexpr uint64_t kDrainNs = 200ull * 1000ull * 1000ull;  // teardown drain limit
// Longest a waiting thread sleeps in one try_wait before it re-checks the
// abort flag and its time limit.
constexpr uint32_t kSleepHintNs = 1000u * 1000u;

enum WaitSite : int {
  kSiteProducerEmpty = 1,
  kSiteMmaAccEmpty = 2,
  kSiteMmaFull = 3,
  kSiteMmaTurn = 5,
  kSiteLoraAuxFull = 6,
  kSiteSfAuxFull = 7,
  kSiteEpiAccFull = 8,
  kSiteSplitFlag = 10,
};

constexpr int kStatusTimeout = -7;       // == SVDQ_ERR_TIMEOUT
constexpr int kStatusWcscaleZero = -11;  // == SVDQ_ERR_WCSCALE_ZERO
constexpr int kStatusLuOverflow = -12;   // == SVDQ_ERR_LU_OVERFLOW

// CG: CTAs per MMA; BN: tile columns; KBI: K blocks (of 256) per main ring
// item.  Larger items halve the fixed per-item costs (one TMA batch, one
// barrier round trip, one scale hand-off per item) at the price of fewer,
// larger ring stages.
template <int CG, int BN, int KBI>
struct Layout {
  static_assert(CG == 1 || CG == 2, "CTA group is 1 or 2");
  static_assert(BN == 128 || BN == 256, "tile_n is 128 or 256");
  static_assert(!(CG == 2 && BN == 128), "a CTA pair uses 256-wide tiles");
  static_assert(KBI == 1 || KBI == 2, "one or two K blocks per ring item");
  static constexpr int kKbi = KBI;
  static constexpr int kSteps = 4 * KBI;                    // K=64 MMA steps per item
  static constexpr int kBNc = BN / CG;                      // B rows held by this CTA
  static constexpr int kATile = kBM * 128;                  // one K block of A: 128 rows x 128 B
  static constexpr int kBTile = kBNc * 128;                 // one K block of B
  static constexpr int kOffA = 0;                           // KBI A tiles
  static constexpr int kOffB = KBI * kATile;                // KBI B tiles
  static constexpr int kOffSFA = kOffB + KBI * kBTile;      // raw [16*KBI groups][128 rows]
  static constexpr int kOffSFB = kOffSFA + 16 * KBI * kBM;  // raw [16*KBI groups][BN] (whole N tile)
  static constexpr int kStageBytes = kOffSFB + 16 * KBI * BN;
  static constexpr int kSfbHalves = BN / 128;
  // LoRA item: LA' [128][32] bf16 and LU' [kBNc][32] bf16 (64-byte rows,
  // 64-byte swizzle), raw LA [128][32] fp32, wcscale [kBNc] bf16.
  static constexpr bool kLuInA = kBNc * 64 <= 8192;
  static constexpr int kLoraLA = kOffA;
  static constexpr int kLoraLU = kLuInA ? kOffA + 8192 : kOffB;
  static constexpr int kLoraRawLA = kLuInA ? kOffB : kOffB + kBNc * 64;
  static constexpr int kLoraWC = kOffSFA;
  // LoRA item with 16-bit LA' (64 ranks, 128-byte rows, 128-byte swizzle):
  // LA' [128][64] over the A tile, LU' [kBNc][64] over the B tile (the same sizes)
  static constexpr int kLora16LA = kOffA;
  static constexpr int kLora16LU = kOffB;
  static_assert(kBM * 128 <= kATile && kBNc * 128 <= kBTile, "64-rank LoRA item fits the stage");
  static_assert(kLoraRawLA + kBM * kLoraRanks * 4 <= kOffSFA, "LoRA item fits the stage");
  static_assert(2 * kBNc <= 16 * kBM, "wcscale fits the scale area");
  static constexpr int kAccStages = (BN == 256) ? 1 : 2;
  static constexpr int kAccCols = kAccStages * BN;
  // tensor-memory scale columns per stage: SFA 4 per K step, then SFB 4*halves per K step
  static constexpr int kSfCols = kSteps * (4 + 4 * kSfbHalves);
  // epilogue, per warp: one 32 x 64 bf16 staging tile (128-byte rows, 128-byte
  // swizzle) and the tile's fp32 wcscale[BN], bias[BN]
  static constexpr int kEpiStageBytes = 32 * 64;
  static constexpr int kEpiBytes = 8 * kEpiStageBytes;
  static constexpr int kWcbBytes = 8 * BN * 4;
  static constexpr int kBarCount = 5 * kMaxStages + 9;
  static constexpr int kBarBytes = 8 * kBarCount + 16;
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned");
  __host__ __device__ static constexpr int epi_offset(int stages) { return stages * kStageBytes; }
  __host__ __device__ static constexpr int wcb_offset(int stages) {
    return epi_offset(stages) + kEpiBytes;
  }
  __host__ __device__ static constexpr int bars_offset(int stages) {
    return wcb_offset(stages) + kWcbBytes;
  }
  __host__ __device__ static constexpr int smem_bytes(int stages) {
    return 1024 /* alignment slack */ + bars_offset(stages) + kBarBytes;
  }
  __host__ __device__ static constexpr int tmem_cols_used(int stages) {
    return kAccCols + stages * kSfCols;
  }
};

struct KParams {
  int M, N, K, R;
  int tiles_m, tiles_n, num_tiles, group_m;
  int k_blocks;     // ceil(K / 256)
  int main_items;   // ceil(k_blocks / K blocks per item)
  int lora_blocks;  // ceil(R / lora_ranks)
  int lora_ranks;   // ranks per LoRA ring item: 32, or 64 with 16-bit LA
  int la16;         // lora_act_in holds 16-bit LA' [M][R] (TMA'd as is, 64 ranks per item)
  int r16;          // R rounded up to 16
  int num_stages;
  int lora_tma;     // R % 8 == 0: LoRA rows arrive by TMA; else direct loads
  int prepacked;    // weights prepacked: scale words [K/64][N], lora_up = LU'
  int act_packed;   // activation scales arrive as words [K/64][M]
  int splits;       // K splits per tile (1: every unit is a whole tile)
  int num_units;    // num_tiles * splits
  float4* partials;       // split-K: fp32 partial tiles of the non-final splits
  unsigned int* flags;    // split-K: one per (tile, non-final split, CTA, epilogue warp);
                          // 0 between launches, 1 while a partial waits to be added
  int debug_fault;
  int ordered;  // the MMA issuers take turns: bit-reproducible accumulation order
  unsigned long long timeout_ns;
  const float* lora_act_in;
  const uint16_t* lora_up;  // bf16 or fp16 bits (the kernel's 16-bit I/O type)
  const uint16_t* wcscale;
  const uint16_t* bias;
  int* status;
};

// Grouped raster over cluster tiles: group_m M-blocks sweep all N-blocks.
__device__ __forceinline__ void tile_coords(const KParams& p, int t, int& mb, int& nb) {
  const int group = p.group_m * p.tiles_n;
  const int gid = t / group;
  const int first_m = gid * p.group_m;
  const int gsz = min(p.tiles_m - first_m, p.group_m);
  const int local = t - gid * group;
  mb = first_m + local % gsz;
  nb = local / gsz;
}

// Main-item visiting order of a tile: tiles that share an A or a B block start
// their K sweep at different items, so the clusters reading one operand block
// at the same time do not all wait on the same first-touch DRAM fetch.  Only
// the fp32 accumulation order changes.
__device__ __forceinline__ int k_rotation(const KParams& p, int mb, int nb) {
  return (7 * mb + 5 * nb) % p.main_items;
}
__device__ __forceinline__ int k_item(const KParams& p, int main_item, int rot) {
  const int it = main_item + rot;
  return it >= p.main_items ? it - p.main_items : it;
}

// A unit of work: one output tile, or one of its `splits` K ranges.  Split s
// covers main K blocks [s * main_items / splits, (s+1) * main_items / splits)
// and split 0 also carries the LoRA items; the last split adds the other
// splits' partial tiles and writes the output.  Units u = tile * splits + s,
// so the units of a tile run on consecutive clusters.
struct Unit {
  int tile, split, lora, kb_begin, nkb;
};
// SK: the kernel instance that splits (the others have splits == 1 built in).
template <bool SK>
__device__ __forceinline__ Unit unit_of(const KParams& p, int u) {
  Unit w;
  if (!SK) {
    w.tile = u;
    w.split = 0;
    w.kb_begin = 0;
    w.nkb = p.main_items;
    w.lora = p.lora_blocks;
    return w;
  }
  w.tile = u / p.splits;
  w.split = u - w.tile * p.splits;
  w.kb_begin = (w.split * p.main_items) / p.splits;
  w.nkb = ((w.split + 1) * p.main_items) / p.splits - w.kb_begin;
  w.lora = (w.split == 0) ? p.lora_blocks : 0;
  return w;
}
// K item of the unit's main item `mi`: a whole tile keeps the per-tile
// rotation, a split walks its own range in order.
template <bool SK>
__device__ __forceinline__ int unit_k_item(const KParams& p, const Unit& w, int mi, int rot) {
  return SK ? w.kb_begin + mi : k_item(p, mi, rot);
}

struct Ctl {
  volatile int* abort_flag;
  int* status;
  unsigned long long timeout_ns;
};

__device__ __noinline__ void report_timeout(int* status, int site) {
  if (atomicCAS(status, 0, kStatusTimeout) == 0) {
    status[1] = site;
    status[2] = static_cast<int>(blockIdx.x);
  }
}

// A LoRA operand the shared accumulator cannot carry: wcscale[n] == 0 with
// R > 0 (LU' = LU / wcscale does not exist, so column n's LoRA term is
// dropped) or LU / wcscale[n] beyond the 16-bit type's range (infinite LU').
// The launch still completes; the first condition recorded in the status
// word wins, with the column.  Warp-collective: `bad` and `n` per lane.
__device__ __noinline__ void report_lora_operand(int* status, int code, int n) {
  if (atomicCAS(status, 0, code) == 0) {
    status[1] = n;
    status[2] = static_cast<int>(blockIdx.x);
  }
}
__device__ __forceinline__ void warp_report_lora(int* status, int code, bool bad, int n) {
  const uint32_t m = __ballot_sync(0xffffffffu, bad);
  if (m != 0u) {
    const int src = __ffs(static_cast<int>(m)) - 1;
    const int col = __shfl_sync(0xffffffffu, n, src);
    if ((threadIdx.x & 31) == 0) report_lora_operand(status, code, col);
  }
}

// Bounded wait for the phase with parity `parity` of a local mbarrier.
// Returns false (and makes every other role of this CTA give up) on expiry or
// if another role already gave up.  CLUSTER selects a cluster-scope acquire,
// needed on the pair leader's barriers that receive the peer's arrivals.
template <bool CLUSTER>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, int site, const Ctl& c) {
  auto probe = [&]() {
    return CLUSTER ? ptx::mbar_try_wait_cluster_sleep(bar, parity, kSleepHintNs)
                   : ptx::mbar_try_wait_sleep(bar, parity, kSleepHintNs);
  };
  if (probe()) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (probe()) return true;
    if (*c.abort_flag) return false;
    if (ptx::globaltimer() - t0 > c.timeout_ns) {
      *c.abort_flag = 1;
      report_timeout(c.status, site);
      return false;
    }
  }
}

template <bool CLUSTER>
__device__ __forceinline__ bool warp_wait_bar(uint32_t bar, uint32_t parity, int site,
                                              const Ctl& c) {
  const bool ok = wait_bar<CLUSTER>(bar, parity, site, c);
  return __all_sync(0xffffffffu, ok);
}

// Split-K: bounded wait until another split has raised its flag (non-zero).
// The waiting split lowers the flag again once it has added the partial, so
// every completed launch leaves its flags at 0: nothing launch-specific is
// compared, and a launch replayed from a CUDA graph waits exactly as a fresh
// one does.
__device__ __forceinline__ bool wait_flag(const unsigned int* f, const Ctl& c) {
  if (ptx::ld_acquire_gpu(f) != 0u) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    __nanosleep(64);
    if (ptx::ld_acquire_gpu(f) != 0u) return true;
    if (*c.abort_flag) return false;
    if (ptx::globaltimer() - t0 > c.timeout_ns) {
      *c.abort_flag = 1;
      report_timeout(c.status, kSiteSplitFlag);
      return false;
    }
  }
}

// Teardown wait: ignores the abort flag, short fixed limit.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > kDrainNs) return;
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The 16-bit I/O type of lora_up, wcscale, bias and the output: bf16 (the
// operator as stated) or IEEE fp16 (the variant the page also measures).
// lo/hi decode the halves of a packed pair, pack rounds two fp32 values (RNE).
template <bool F16>
struct H16 {
  static __device__ __forceinline__ float one(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }
  static __device__ __forceinline__ float lo(uint32_t w) { return bf16_lo(w); }
  static __device__ __forceinline__ float hi(uint32_t w) { return bf16_hi(w); }
  static __device__ __forceinline__ uint32_t pack(float a, float b) { return ptx::pack_bf16x2(a, b); }
  static constexpr uint32_t kOnes = 0x3F803F80u;  // (1.0, 1.0)
};
template <>
struct H16<true> {
  static __device__ __forceinline__ float one(uint16_t b) {
    return __half2float(__ushort_as_half(b));
  }
  static __device__ __forceinline__ float lo(uint32_t w) { return one(uint16_t(w & 0xFFFFu)); }
  static __device__ __forceinline__ float hi(uint32_t w) { return one(uint16_t(w >> 16)); }
  static __device__ __forceinline__ uint32_t pack(float a, float b) { return ptx::pack_f16x2(a, b); }
  static constexpr uint32_t kOnes = 0x3C003C00u;
};

// Non-zero iff either half of a packed 16-bit pair has an all-ones exponent
// (infinite or NaN); branch-free for the hot loops.  Adding the exponent's lowest bit to
// the magnitude carries into bit 15 exactly then; no carry crosses halves.
template <bool F16>
__device__ __forceinline__ uint32_t nonfinite16_bits(uint32_t w) {
  constexpr uint32_t kInc = F16 ? 0x04000400u : 0x00800080u;
  return ((w & 0x7FFF7FFFu) + kInc) & 0x80008000u;
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// Matrix row (or column) offset held by tile row r under the row-quad order:
// within each 128-row block, row a + 32b holds offset 4a + b.
__device__ __forceinline__ int quad_row(int r) {
  return (r & ~127) | (4 * (r & 31)) | ((r >> 5) & 3);
}

// Scale words of one K step (4 groups) for one 128-row block.  `raw` points at
// group 0 of the block in a raw [group][row] scale box with `pitch` bytes per
// group; lane a gets w[b] = the 4 group scales (byte g = group g) of block row
// 4a + b, the word tensor-memory lane a, column b takes.
__device__ __forceinline__ void sf_words(const uint8_t* raw, int pitch, int lane, uint32_t* w) {
  const uint8_t* p = raw + 4 * lane;
  const uint32_t g0 = *reinterpret_cast<const uint32_t*>(p);
  const uint32_t g1 = *reinterpret_cast<const uint32_t*>(p + pitch);
  const uint32_t g2 = *reinterpret_cast<const uint32_t*>(p + 2 * pitch);
  const uint32_t g3 = *reinterpret_cast<const uint32_t*>(p + 3 * pitch);
  // 4x4 byte transpose: byte b of group g -> byte g of word b
  const uint32_t t0 = __byte_perm(g0, g1, 0x5140);
  const uint32_t t1 = __byte_perm(g0, g1, 0x7362);
  const uint32_t t2 = __byte_perm(g2, g3, 0x5140);
  const uint32_t t3 = __byte_perm(g2, g3, 0x7362);
  w[0] = __byte_perm(t0, t2, 0x5410);
  w[1] = __byte_perm(t0, t2, 0x7632);
  w[2] = __byte_perm(t1, t3, 0x5410);
  w[3] = __byte_perm(t1, t3, 0x7632);
}

// One 32-column group of packed 16-bit outputs (v[2k], v[2k+1] = columns
// 4k .. 4k+3) as row `lane` of a 32 x 32 staging tile with 64-byte rows and
// the 64-byte swizzle: 16-byte chunk j holds columns 8j .. 8j+7 at chunk
// index j XOR bits 1..2 of the row.
__device__ __forceinline__ void stage_row(uint8_t* stg, int lane, const uint32_t* v) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(stg + 64 * lane + ((j ^ ((lane >> 1) & 3)) << 4)) =
        make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}

// Byte offset of 16-byte chunk `chunk` (0..3) of row `row` in a K-major tile
// with 64-byte rows and the 64-byte swizzle.
__device__ __forceinline__ int sw64_offset(int row, int chunk) {
  return row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);
}

// LA' rows r0 .. r0+31 from the TMA-staged raw fp32 rows [128][32] (already in
// row-quad order): lane reads 4 consecutive floats of a row, writes 4 bf16
// (half a 16-byte chunk).
template <bool F16>
__device__ __forceinline__ void lora_la_from_smem(uint8_t* dst, const uint8_t* raw, int r0,
                                                  int lane) {
  const int c = lane & 7;  // 16-byte piece of the 128-byte raw row
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int row = r0 + it * 4 + (lane >> 3);
    const float4 v = *reinterpret_cast<const float4*>(raw + row * 128 + 16 * c);
    uint2 pk;
    pk.x = H16<F16>::pack(v.x, v.y);
    pk.y = H16<F16>::pack(v.z, v.w);
    *reinterpret_cast<uint2*>(dst + sw64_offset(row, c >> 1) + 8 * (c & 1)) = pk;
  }
}

// LU' rows [r0, r0 + NR) of a LoRA item in place: tile row r (column n =
// n_cta + quad_row(r)) times 1/wcscale[n] (fp32 product, 16-bit RNE); the
// staged wcscale is in plain column order.  ROWB-byte rows: 64 (32 ranks,
// 64-byte swizzle) or 128 (64 ranks, 128-byte swizzle); a row's 16-byte chunks
// stay in the row, so whole rows scale alike whatever the swizzle.  Rows
// outside N (zero-filled) stay zero.  inv[t] holds the reciprocal of row
// r0 + lane + 32t (0 beyond NR, outside N or for a zero wcscale); it is
// computed on a tile's first LoRA item (`fresh`) and kept for the others,
// which carry the same columns.  zero_col / bad_col (-1 if none): a column
// with a zero wcscale (reported on the fresh item), a column whose LU' is not
// finite; the caller reports them once its ring arrival is made (the checks
// are branch-free, off the ring's path).
template <int NR, int ROWB, bool F16>
__device__ __forceinline__ void lora_lu_scale(uint8_t* lu, const uint8_t* wc, int n_cta, int N,
                                              int r0, int lane, bool fresh, float* inv,
                                              int& zero_col, int& bad_col) {
  using H = H16<F16>;
  constexpr int kCpr = ROWB / 16;  // 16-byte chunks per row
  constexpr int kRpi = 32 / kCpr;  // rows per pass of the warp
  static_assert(NR % kRpi == 0, "whole passes");
  if (fresh) {
#pragma unroll
    for (int t = 0; t < (NR + 31) / 32; ++t) {
      const int rl = lane + 32 * t;
      const int off = quad_row(r0 + rl);
      const bool mine = rl < NR;
      const float w = mine ? H::one(*reinterpret_cast<const uint16_t*>(wc + 2 * off)) : 0.f;
      const bool in = mine && n_cta + off < N;
      inv[t] = (in && w != 0.f) ? __frcp_rn(w) : 0.f;
      zero_col = (in && w == 0.f) ? n_cta + off : zero_col;
    }
  }
  const int pc = lane % kCpr;
  uint32_t any_bad = 0u;
  int bad_row = 0;
#pragma unroll
  for (int it = 0; it < NR / kRpi; ++it) {
    const int rl = it * kRpi + lane / kCpr;
    const int row = r0 + rl;
    // rows of one pass share a 32-row block of inv
    const float s = __shfl_sync(0xffffffffu, inv[(it * kRpi) / 32], rl % 32);
    uint4 x = *reinterpret_cast<uint4*>(lu + row * ROWB + 16 * pc);
    x.x = H::pack(__fmul_rn(H::lo(x.x), s), __fmul_rn(H::hi(x.x), s));
    x.y = H::pack(__fmul_rn(H::lo(x.y), s), __fmul_rn(H::hi(x.y), s));
    x.z = H::pack(__fmul_rn(H::lo(x.z), s), __fmul_rn(H::hi(x.z), s));
    x.w = H::pack(__fmul_rn(H::lo(x.w), s), __fmul_rn(H::hi(x.w), s));
    const uint32_t b = nonfinite16_bits<F16>(x.x) | nonfinite16_bits<F16>(x.y) |
                       nonfinite16_bits<F16>(x.z) | nonfinite16_bits<F16>(x.w);
    any_bad |= b;
    bad_row = b ? row : bad_row;
    *reinterpret_cast<uint4*>(lu + row * ROWB + 16 * pc) = x;
  }
  bad_col = any_bad ? n_cta + quad_row(bad_row) : bad_col;
}

// Direct-load LoRA operands (used when R is not a multiple of 8, so LoRA rows
// are not 16-byte strided for TMA): LA' tile row r holds matrix row m_cta +
// quad_row(r), LU' tile row r column n_cta + quad_row(r); ranks 32*blk ..
// 32*blk+31, zero outside [M|N, R).  Rows r0 .. r0+NR-1.
template <int NR, bool F16>
__device__ __forceinline__ void lora_la_direct(uint8_t* dst, const KParams& p, int m_cta, int blk,
                                               int r0, int lane) {
  const int chunk = lane & 3;
  const int k0 = blk * kLoraRanks + chunk * 8;
  for (int it = 0; it < NR / 8; ++it) {
    const int row = r0 + it * 8 + (lane >> 2);
    const int m = m_cta + quad_row(row);
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      v[q] = (m < p.M && k0 + q < p.R) ? __ldg(p.lora_act_in + (size_t)m * p.R + k0 + q) : 0.f;
    uint4 pk;
    pk.x = H16<F16>::pack(v[0], v[1]);
    pk.y = H16<F16>::pack(v[2], v[3]);
    pk.z = H16<F16>::pack(v[4], v[5]);
    pk.w = H16<F16>::pack(v[6], v[7]);
    *reinterpret_cast<uint4*>(dst + sw64_offset(row, chunk)) = pk;
  }
}

// `wc` is NULL for a prepacked LU' (already divided) or an absent wcscale.
// zero_col / bad_col as for lora_lu_scale_smem.
template <int NR, bool F16>
__device__ __forceinline__ void lora_lu_direct(uint8_t* dst, const KParams& p,
                                               const uint16_t* wc, int n_cta, int blk, int r0,
                                               int lane, int& zero_col, int& bad_col) {
  const int chunk = lane & 3;
  const int k0 = blk * kLoraRanks + chunk * 8;
  const uint16_t* lu = p.lora_up;
  for (int it = 0; it < NR / 8; ++it) {
    const int row = r0 + it * 8 + (lane >> 2);
    const int n = n_cta + quad_row(row);
    float inv = 0.f;
    if (n < p.N) {
      const float w = wc ? H16<F16>::one(__ldg(wc + n)) : 1.f;
      inv = (w != 0.f) ? __frcp_rn(w) : 0.f;
      zero_col = (w == 0.f) ? n : zero_col;
    }
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      v[q] = (n < p.N && k0 + q < p.R)
                 ? __fmul_rn(H16<F16>::one(__ldg(lu + (size_t)n * p.R + k0 + q)), inv)
                 : 0.f;
    uint4 pk;
    pk.x = H16<F16>::pack(v[0], v[1]);
    pk.y = H16<F16>::pack(v[2], v[3]);
    pk.z = H16<F16>::pack(v[4], v[5]);
    pk.w = H16<F16>::pack(v[6], v[7]);
    const uint32_t b = nonfinite16_bits<F16>(pk.x) | nonfinite16_bits<F16>(pk.y) |
                       nonfinite16_bits<F16>(pk.z) | nonfinite16_bits<F16>(pk.w);
    bad_col = b ? n : bad_col;
    *reinterpret_cast<uint4*>(dst + sw64_offset(row, chunk)) = pk;
  }
}

template <int CG, int BN, int KBI, bool F16, bool SK>
__global__ void __launch_bounds__(kThreads, 1)
    svdq_w4a4_kernel(const __grid_constant__ CUtensorMap tm_act,
                     const __grid_constant__ CUtensorMap tm_wgt,
                     const __grid_constant__ CUtensorMap tm_sfa,
                     const __grid_constant__ CUtensorMap tm_sfb,
                     const __grid_constant__ CUtensorMap tm_la,
                     const __grid_constant__ CUtensorMap tm_lu,
                     const __grid_constant__ CUtensorMap tm_wc,
                     const __grid_constant__ CUtensorMap tm_out, const KParams p) {
  using L = Layout<CG, BN, KBI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = static_cast<int>(threadIdx.x) / 32;
  const int lane = static_cast<int>(threadIdx.x) % 32;
  const int S = p.num_stages;
  const uint32_t rank = (CG == 2) ? ptx::cluster_ctarank() : 0u;
  const bool leader = (rank == 0);
  const int cluster_id = static_cast<int>(blockIdx.x) / CG;
  const int num_clusters = static_cast<int>(gridDim.x) / CG;

  uint8_t* bar_area = smem + L::bars_offset(S);
  const uint32_t bar0 = ptx::smem_u32(bar_area);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
  auto auxfull = [&](int s) { return bar0 + 8u * (2 * kMaxStages + s); };
  auto acc_full = [&](int a) { return bar0 + 8u * (5 * kMaxStages + a); };
  auto acc_empty = [&](int a) { return bar0 + 8u * (5 * kMaxStages + 2 + a); };
  const uint32_t never = bar0 + 8u * (5 * kMaxStages + 4);  // no role arrives on it
  auto drain = [&](uint32_t e) { return bar0 + 8u * (5 * kMaxStages + 5 + e); };
  // issuer e arrives on turn(e) once it has issued an item's MMAs
  auto turn = [&](uint32_t e) { return bar0 + 8u * (5 * kMaxStages + 7 + e); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 8 * L::kBarCount);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const Ctl ctl{abort_flag, p.status, p.timeout_ns};
  // Barriers the leader owns, addressed from either CTA of the pair.
  auto to_leader = [&](uint32_t local_bar) {
    return CG == 2 ? ptx::mapa(local_bar, 0) : local_bar;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // the leader's count: its scale producer, then the scale feeders and
      // LoRA builders of every CTA of the group (their shared-memory and
      // tensor-memory writes are done); the act / wgt bytes come as transactions
      ptx::mbar_init(full(s), 1 + 6 * CG);
      ptx::mbar_init(empty(s), 2);  // the owning issuer's commit, the other's arrival
      ptx::mbar_init(auxfull(s), 3);  // one arrival per producer
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(acc_full(a), 2);          // one commit per MMA issuer
      ptx::mbar_init(acc_empty(a), 8 * CG);    // the epilogue warps of the group
    }
    ptx::mbar_init(never, 1);
    ptx::mbar_init(drain(0), 1);
    ptx::mbar_init(drain(1), 1);
    ptx::mbar_init(turn(0), 1);
    ptx::mbar_init(turn(1), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tm_act);
    ptx::prefetch_tmap(&tm_wgt);
    ptx::prefetch_tmap(&tm_sfa);
    ptx::prefetch_tmap(&tm_sfb);
  }
  if (warp == 1) {
    if (CG == 2) {
      ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (CG == 2) ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  // Launched with programmatic stream serialisation: the set-up above may
  // overlap the tail of the previous kernel in the stream, but no global
  // memory is read or written before that kernel has completed.  Kernels
  // launched after this one may be scheduled from here on (they wait the same
  // way before touching memory).
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();

  if (warp == 0 || warp == 12 || warp == 13) {
    // ------------------------------------------------------------ producers
    if (lane == 0) {
      // role 0: scale boxes, LoRA rows, the byte counts; 1: act tiles; 2: wgt tiles
      const int role = warp == 0 ? 0 : warp - 11;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint32_t main_aux_bytes = 16 * KBI * (kBM + BN);
      // the LoRA item stages wcscale only to divide LU by it in place
      const bool stage_wc = p.wcscale != nullptr && !p.prepacked;
      const uint32_t lora_aux_bytes =
          p.la16 ? kBM * 128 + L::kBNc * 128 + (stage_wc ? 2 * L::kBNc : 0)
                 : kBM * kLoraRanks * 4 + L::kBNc * 64 + (stage_wc ? 2 * L::kBNc : 0);
      for (int u = cluster_id; ok && u < p.num_units; u += num_clusters) {
        const Unit w = unit_of<SK>(p, u);
        const int t = w.tile;
        const int n_items = w.lora + w.nkb;
        int mb, nb;
        tile_coords(p, t, mb, nb);
        const int m0 = mb * kBM * CG, n0 = nb * BN;
        const int m_cta = m0 + kBM * static_cast<int>(rank);
        const int n_cta = n0 + L::kBNc * static_cast<int>(rank);
        const int rot = k_rotation(p, mb, nb);
        for (int i = 0; i < n_items; ++i) {
          if (!wait_bar<false>(empty(stage), phase ^ 1u, kSiteProducerEmpty, ctl)) {
            ok = false;
            break;
          }
          const uint32_t st = sbase + stage * L::kStageBytes;
          const uint32_t ab = auxfull(stage);
          if (role != 0) {
            // Every producer signs every item on the stage's aux barrier, so no
            // item is consumed before all three have passed their wait for it:
            // none can fall two phases behind (or run two ahead) on a barrier
            // it tracks by parity, LoRA items (no act / wgt loads) included.
            ptx::mbar_arrive(ab);
          }
          if (i < w.lora) {
            if (role == 0) {
              if (p.la16) {
                // 64 ranks of 16-bit LA' and LU (128-byte swizzle), as they come
                ptx::mbar_arrive_expect_tx(ab, lora_aux_bytes);
                ptx::tma_load_3d(st + L::kLora16LA, &tm_la, ab, 64 * i, m_cta / 4, 0);
#pragma unroll
                for (int h = 0; h < L::kBNc / 128; ++h)
                  ptx::tma_load_3d(st + L::kLora16LU + 16384 * h, &tm_lu, ab, 64 * i,
                                   (n_cta + 128 * h) / 4, 0);
                if (stage_wc) ptx::tma_load_1d(st + L::kLoraWC, &tm_wc, ab, n_cta);
              } else if (p.lora_tma) {
                ptx::mbar_arrive_expect_tx(ab, lora_aux_bytes);
                ptx::tma_load_3d(st + L::kLoraRawLA, &tm_la, ab, kLoraRanks * i, m_cta / 4, 0);
#pragma unroll
                for (int h = 0; h < L::kBNc / 128; ++h)
                  ptx::tma_load_3d(st + L::kLoraLU + 8192 * h, &tm_lu, ab, kLoraRanks * i,
                                   (n_cta + 128 * h) / 4, 0);
                if (stage_wc) ptx::tma_load_1d(st + L::kLoraWC, &tm_wc, ab, n_cta);
              } else {
                ptx::mbar_arrive(ab);
              }
              if (leader) ptx::mbar_arrive(full(stage));
            }
          } else {
            const int kb0 = KBI * unit_k_item<SK>(p, w, i - w.lora, rot);
            const int nkb = min(KBI, p.k_blocks - kb0);
            if (role == 0) {
              ptx::mbar_arrive_expect_tx(ab, main_aux_bytes);
              // raw scales: 16 group rows per K block; packed words: 4 step rows
              ptx::tma_load_2d(st + L::kOffSFA, &tm_sfa, ab, m_cta,
                               kb0 * (p.act_packed ? 4 : 16));
              ptx::tma_load_2d(st + L::kOffSFB, &tm_sfb, ab, n0, kb0 * (p.prepacked ? 4 : 16));
              // The act / wgt loads of this item may land before this count
              // (the transaction count runs negative meanwhile); the phase
              // cannot complete before this arrival.
              if (leader)
                ptx::mbar_arrive_expect_tx(full(stage), CG * nkb * (L::kATile + L::kBTile));
            } else {
              const uint32_t fb = to_leader(full(stage));
              for (int kk = 0; kk < nkb; ++kk) {
                const int kx = (kb0 + kk) * 128;
                if (role == 1) {
                  const uint32_t da = st + L::kOffA + kk * L::kATile;
                  if (CG == 2)
                    ptx::tma_load_3d_pair(da, &tm_act, fb, kx, m_cta / 4, 0);
                  else
                    ptx::tma_load_3d(da, &tm_act, fb, kx, m_cta / 4, 0);
                } else {
#pragma unroll
                  for (int h = 0; h < L::kBNc / 128; ++h) {
                    const uint32_t db = st + L::kOffB + kk * L::kBTile + 16384 * h;
                    const int y = (n_cta + 128 * h) / 4;
                    if (CG == 2)
                      ptx::tma_load_3d_pair(db, &tm_wgt, fb, kx, y, 0);
                    else
                      ptx::tma_load_3d(db, &tm_wgt, fb, kx, y, 0);
                  }
                }
              }
            }
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // On the normal path every load has been consumed before the teardown
      // barrier.  After an abort a load may still be landing in this CTA's
      // shared memory (or signalling the pair leader): give it a fixed grace
      // period before the CTA can exit.
      if (!ok) {
        const uint64_t t0 = ptx::globaltimer();
        while (ptx::globaltimer() - t0 < 200000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 14) {
    // ------------------------------------------------------------ MMA issuers
    // Two threads of the leader CTA share the ring: issuer e issues the MMAs
    // of items j with j % 2 == e (j counts items over all tiles), so one
    // thread's per-item cost (barrier wait, descriptors, commit) is spread
    // over two items' worth of tensor-core time.  Both wait on every item's
    // full barrier in order and signs every item's release, so neither can
    // fall two phases behind on a barrier it tracks by parity.
    // Every MMA accumulates: the epilogue zeroes the accumulator when it has
    // read it (and once before the first tile), so no MMA waits for another to
    // complete.  The issuers still take turns: after issuing item j's MMAs,
    // its owner executes tcgen05.fence::before_thread_sync and arrives on its
    // turn barrier (a CTA-scope release); the other issuer waits on that
    // barrier (acquire) and executes tcgen05.fence::after_thread_sync before
    // issuing item j + 1.  That orders the MMAs of successive items in ring
    // order without waiting for any of them to complete, so the fp32
    // accumulation order, and with it every output bit, is fixed.
    if (lane == 0 && leader) {
      const uint32_t me = warp == 1 ? 0u : 1u;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t j = 0;
      bool ok = true;
      int tile_iter = 0;
      constexpr uint32_t kIdescMain = ptx::idesc_mxf4nvf4(kBM * CG, BN);
      constexpr uint32_t kIdescLora =
          F16 ? ptx::idesc_f16_f32(kBM * CG, BN) : ptx::idesc_bf16_f32(kBM * CG, BN);
      const uint64_t desc_a0 = ptx::desc_kmajor_sw128(sbase + L::kOffA);
      const uint64_t desc_b0 = ptx::desc_kmajor_sw128(sbase + L::kOffB);
      const bool k_ragged = (p.K % kBK) != 0;  // the last K block is partial
      for (int u = cluster_id; ok && u < p.num_units; u += num_clusters, ++tile_iter) {
        const Unit w = unit_of<SK>(p, u);
        const int t = w.tile;
        const int n_items = w.lora + w.nkb;
        int mb, nb;
        tile_coords(p, t, mb, nb);
        const int rot = k_rotation(p, mb, nb);
        const int acc_stage = tile_iter % L::kAccStages;
        const uint32_t acc_phase = static_cast<uint32_t>(tile_iter / L::kAccStages) & 1u;
        // A zeroed accumulator: the epilogue read this buffer's previous tile
        // (or cleared it at start).  debug_fault waits on a barrier no role
        // arrives on instead, so the wait must expire.
        const bool got = p.debug_fault ? wait_bar<false>(never, 0u, kSiteMmaAccEmpty, ctl)
                                       : wait_bar<CG == 2>(acc_empty(acc_stage), acc_phase,
                                                           kSiteMmaAccEmpty, ctl);
        if (!got) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc_stage * BN);
        // LoRA items, then K-block items: one loop each, compiled apart
        auto run_items = [&](auto lora_tag, int i0, int i1) {
          constexpr bool kLoraItems = decltype(lora_tag)::value;
          for (int i = i0; ok && i < i1; ++i, ++j) {
            if (!wait_bar<CG == 2>(full(stage), phase, kSiteMmaFull, ctl)) {
              ok = false;
              break;
            }
            if ((j & 1u) == me) {
              // Everything the MMAs need is computed before this issuer's turn.
              const uint32_t st = sbase + stage * L::kStageBytes;
              int nsteps;  // MMAs of this item
              if constexpr (kLoraItems) {
                nsteps = min(p.lora_ranks / 16, (p.r16 - p.lora_ranks * i) / 16);
              } else {
                // K=64 steps present in this item (the last K block may be partial)
                nsteps = L::kSteps;
                if (k_ragged) {
                  const int kb0 = KBI * unit_k_item<SK>(p, w, i - w.lora, rot);
                  nsteps = min(L::kSteps, (p.K - kb0 * kBK) / 64);
                }
              }
              const uint32_t sf =
                  tmem_base + static_cast<uint32_t>(L::kAccCols + stage * L::kSfCols);
              // descriptors of this stage's first K step; a step advances the
              // start address (descriptor units of 16 bytes)
              const uint64_t soff = static_cast<uint64_t>((stage * L::kStageBytes) >> 4);
              const uint64_t ad0 = desc_a0 + soff, bd0 = desc_b0 + soff;
              auto step = [&](int ks) {
                const int kk = ks >> 2, s4 = ks & 3;
                const uint64_t ad = ad0 + static_cast<uint64_t>((kk * L::kATile + 32 * s4) >> 4);
                const uint64_t bd = bd0 + static_cast<uint64_t>((kk * L::kBTile + 32 * s4) >> 4);
                const uint32_t sfa = sf + 4 * ks;
                const uint32_t sfb = sf + 4 * L::kSteps + 4 * ks * L::kSfbHalves;
                if (CG == 2)
                  ptx::mma_mxf4nvf4_pair(d_tmem, ad, bd, kIdescMain, sfa, sfb, 1u);
                else
                  ptx::mma_mxf4nvf4(d_tmem, ad, bd, kIdescMain, sfa, sfb, 1u);
              };
              // Items reach the tensor core in ring order: the fp32 accumulation
              // order, and with it every output bit, is the same on every call
              // (unless the caller relaxed the order for the last few percent).
              // Item j - 1 is the other issuer's ((j - 1) >> 1)-th item, i.e. the
              // completion of that phase of its turn barrier.
              if (p.ordered && j > 0 &&
                  !wait_bar<false>(turn(me ^ 1u), ((j - 1u) >> 1) & 1u, kSiteMmaTurn, ctl)) {
                ok = false;
                break;
              }
              ptx::tc_fence_after();
              if constexpr (kLoraItems) {
                for (int s = 0; s < nsteps; ++s) {
                  const uint64_t ad = p.la16 ? ptx::desc_kmajor_sw128(st + L::kLora16LA + 32 * s)
                                             : ptx::desc_kmajor_sw64(st + L::kLoraLA + 32 * s);
                  const uint64_t bd = p.la16 ? ptx::desc_kmajor_sw128(st + L::kLora16LU + 32 * s)
                                             : ptx::desc_kmajor_sw64(st + L::kLoraLU + 32 * s);
                  if (CG == 2)
                    ptx::mma_bf16_pair(d_tmem, ad, bd, kIdescLora, 1u);
                  else
                    ptx::mma_bf16(d_tmem, ad, bd, kIdescLora, 1u);
                }
              } else if (nsteps == L::kSteps) {
#pragma unroll
                for (int ks = 0; ks < L::kSteps; ++ks) step(ks);
              } else {
                for (int ks = 0; ks < nsteps; ++ks) step(ks);
              }
              // Hand the turn over (see above).
              if (p.ordered) {
                ptx::tc_fence_before();
                ptx::mbar_arrive(turn(me));
              }
              if (CG == 2)
                ptx::mma_commit_pair_multicast(empty(stage), 3);
              else
                ptx::mma_commit(empty(stage));
            } else {
              // Not this issuer's item: sign the stage's release anyway, so the
              // producers refill it only after both issuers have passed its
              // full barrier (neither can then be lapped on that barrier).
              ptx::mbar_arrive(empty(stage));
              if (CG == 2) ptx::mbar_arrive_remote(ptx::mapa(empty(stage), 1));
            }
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
        };
        run_items(std::true_type{}, 0, w.lora);
        run_items(std::false_type{}, w.lora, n_items);
        if (!ok) break;
        // this issuer's share of the tile is done (the epilogue waits for both)
        if (CG == 2)
          ptx::mma_commit_pair_multicast(acc_full(acc_stage), 3);
        else
          ptx::mma_commit(acc_full(acc_stage));
      }
      // Every tcgen05 operation issued here completes before tensor memory is freed.
      if (CG == 2)
        ptx::mma_commit_pair(drain(me));
      else
        ptx::mma_commit(drain(me));
      drain_wait(drain(me), 0);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------ LoRA operand builders
    // A unit's LoRA items come first, then its K-block items (nothing to build)
    constexpr int kLuRowsB = L::kBNc / 4;  // LU' rows scaled per builder warp
    int stage = 0;
    uint32_t phase = 0;
    const uint32_t full_bar0 = to_leader(full(0));
    bool ok = true;
    for (int u = cluster_id; ok && u < p.num_units; u += num_clusters) {
      const Unit w = unit_of<SK>(p, u);
      const int t = w.tile;
      int mb, nb;
      tile_coords(p, t, mb, nb);
      const int n_cta = nb * BN + L::kBNc * static_cast<int>(rank);
      float lu_inv[(kLuRowsB + 31) / 32];
      for (int i = 0; i < w.lora; ++i) {
        if (!warp_wait_bar<false>(auxfull(stage), phase, kSiteLoraAuxFull, ctl)) {
          ok = false;
          break;
        }
        int zero_col = -1, bad_col = -1;
        uint8_t* st = smem + stage * L::kStageBytes;
        if (!p.lora_tma && !p.la16) {
          // direct loads (R not a multiple of 8): LU' rows [h kBNc/2, (h+1) kBNc/2)
          lora_lu_direct<L::kBNc / 2, F16>(st + L::kLoraLU, p,
                                           p.prepacked ? nullptr : p.wcscale, n_cta, i,
                                           (warp - 2) * (L::kBNc / 2), lane, zero_col, bad_col);
        } else if (p.wcscale != nullptr && !p.prepacked) {
          // LU / wcscale in place: rows [0, kBNc/2) here (a quarter each), the
          // rest by the scale feeders
          const int r0 = (warp - 2) * kLuRowsB;
          if (p.la16)
            lora_lu_scale<kLuRowsB, 128, F16>(st + L::kLora16LU, st + L::kLoraWC, n_cta, p.N,
                                              r0, lane, i == 0, lu_inv, zero_col, bad_col);
          else
            lora_lu_scale<kLuRowsB, 64, F16>(st + L::kLoraLU, st + L::kLoraWC, n_cta, p.N, r0,
                                             lane, i == 0, lu_inv, zero_col, bad_col);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        // The pair peer's LoRA rows are generic shared-memory writes that the
        // leader's MMA reads: the proxy fence above orders them before this
        // arrival (CTA-scope release, as for every other arrival here).
        if (lane == 0) ptx::mbar_arrive_remote(full_bar0 + 8u * stage);
        // LoRA operands the accumulator cannot carry, reported after the
        // arrival so that the ring does not wait for it
        warp_report_lora(p.status, kStatusWcscaleZero, zero_col >= 0, zero_col);
        warp_report_lora(p.status, kStatusLuOverflow, bad_col >= 0, bad_col);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      for (int j = 0; ok && j < w.nkb; ++j) {
        if (!warp_wait_bar<false>(auxfull(stage), phase, kSiteLoraAuxFull, ctl)) {
          ok = false;
          break;
        }
        if (lane == 0) ptx::mbar_arrive_remote(full_bar0 + 8u * stage);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp < 8 || warp >= 15) {
    // ------------------------------------------------------------ epilogue
    // Two warps per tensor-memory lane quadrant: warps 4..7 take the tile's
    // first half of the column groups, warps 15..18 the second half.
    const int q = warp & 3;  // tensor-memory lane quadrant of this warp
    const int eh = warp >= 15 ? 1 : 0;
    const int ew = 4 * eh + q;  // epilogue warp index
    constexpr int kGroups = BN / 32;
    constexpr int kHalfG = kGroups / 2;
    const int g0 = eh * kHalfG;  // this warp's first column group
    using H = H16<F16>;
    const uint16_t* wcg = p.wcscale;
    const uint16_t* big = p.bias;
    uint8_t* stg = smem + L::epi_offset(S) + ew * L::kEpiStageBytes;
    // this warp's half of the tile's wcscale, bias as fp32: wb[c], wb[BN/2 + c]
    float* wb = reinterpret_cast<float*>(smem + L::wcb_offset(S) + ew * (4 * BN));
    const uint32_t acc_empty0 = to_leader(acc_empty(0));
    const uint32_t zero8[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    const uint32_t lane_q = static_cast<uint32_t>(32 * q) << 16;
    // The MMAs only accumulate: clear every accumulator buffer once before the
    // first tile (each warp its own lanes and column groups), then hand them
    // to the MMA issuers.
    for (int a = 0; a < L::kAccStages; ++a)
      for (int g = g0; g < g0 + kHalfG; ++g)
        for (int b = 0; b < 4; ++b)
          ptx::tmem_st_32x32b_x8(tmem_base + lane_q +
                                     static_cast<uint32_t>(a * BN + 128 * (g >> 2) + 8 * (g & 3) +
                                                           32 * b),
                                 zero8);
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0)
      for (int a = 0; a < L::kAccStages; ++a) ptx::mbar_arrive_remote(acc_empty0 + 8u * a);
    int tile_iter = 0;
    for (int u = cluster_id; u < p.num_units; u += num_clusters, ++tile_iter) {
      const Unit w = unit_of<SK>(p, u);
      const int t = w.tile;
      int mb, nb;
      tile_coords(p, t, mb, nb);
      const int m_cta = mb * kBM * CG + kBM * static_cast<int>(rank);
      const int n0 = nb * BN;
      // This tile's wcscale / bias (this warp's half) as fp32 in this warp's
      // own buffer (no other warp reads it; the previous tile's reads are
      // behind us in program order).
      if (lane < BN / 16) {
        const int c = 8 * lane;
        const int n = n0 + 32 * g0 + c;
        uint4 wv = make_uint4(H::kOnes, H::kOnes, H::kOnes, H::kOnes);  // 1.0
        uint4 bv = make_uint4(0u, 0u, 0u, 0u);
        if (n < p.N) {
          if (wcg) wv = __ldg(reinterpret_cast<const uint4*>(wcg + n));
          if (big) bv = __ldg(reinterpret_cast<const uint4*>(big + n));
        }
        const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w}, b4[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          *reinterpret_cast<float4*>(wb + c + 4 * i) =
              make_float4(H::lo(w4[2 * i]), H::hi(w4[2 * i]), H::lo(w4[2 * i + 1]),
                          H::hi(w4[2 * i + 1]));
          *reinterpret_cast<float4*>(wb + BN / 2 + c + 4 * i) =
              make_float4(H::lo(b4[2 * i]), H::hi(b4[2 * i]), H::lo(b4[2 * i + 1]),
                          H::hi(b4[2 * i + 1]));
        }
      }
      __syncwarp();
      const int acc_stage = tile_iter % L::kAccStages;
      const uint32_t acc_phase = static_cast<uint32_t>(tile_iter / L::kAccStages) & 1u;
      if (!warp_wait_bar<false>(acc_full(acc_stage), acc_phase, kSiteEpiAccFull, ctl)) break;
      ptx::tc_fence_after();
      // Split-K: a non-final split stores its fp32 partial tile (no affine)
      // and raises its flag; the final split waits for the other splits'
      // flags and adds their partials before the affine.  Partial slot
      // (tile, split, CTA) holds this warp's rows as float4 [group][k][lane]
      // (coalesced: lane-consecutive 16-byte pieces).
      const bool write_partial = SK && w.split < p.splits - 1;
      const bool add_partials = SK && !write_partial;
      // slot of (tile, split sp, CTA) = (t (splits - 1) + sp) CG + rank
      const size_t slot0 = static_cast<size_t>(t) * static_cast<size_t>(p.splits - 1) * CG + rank;
      constexpr size_t kSlotF4 = static_cast<size_t>(kBM) * BN / 4;  // float4 per slot
      const float4* part0 = p.partials + slot0 * kSlotF4 + (q * kGroups * 8) * 32 + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                             static_cast<uint32_t>(acc_stage * BN);
      auto gcol = [&](int g) { return taddr + 128 * (g >> 2) + 8 * (g & 3); };
      // one flag per (slot, epilogue warp)
      auto flag = [&](int sp) { return p.flags + (slot0 + static_cast<size_t>(sp) * CG) * 8 + ew; };
      if (write_partial) {
        for (int g = g0; g < g0 + kHalfG; ++g) {
          uint32_t v[4][8];
#pragma unroll
          for (int b = 0; b < 4; ++b) ptx::tmem_ld_32x32b_x8(gcol(g) + 32 * b, v[b]);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int b = 0; b < 4; ++b) ptx::tmem_st_32x32b_x8(gcol(g) + 32 * b, zero8);
          float4* dst = const_cast<float4*>(part0) + static_cast<size_t>(w.split) * CG * kSlotF4 +
                        g * 256;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            __stcg(dst + 32 * k, make_float4(__uint_as_float(v[0][k]), __uint_as_float(v[1][k]),
                                             __uint_as_float(v[2][k]), __uint_as_float(v[3][k])));
        }
        // read and cleared: release the accumulator, then publish the partial
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_remote(acc_empty0 + 8u * acc_stage);
        __threadfence();  // every lane's partial stores are visible device-wide ...
        __syncwarp();     // ... before lane 0 raises the flag
        if (lane == 0) ptx::st_release_gpu(flag(w.split), 1u);
        continue;
      }
      if (add_partials) {
        bool got = true;
        for (int sp = 0; sp < p.splits - 1 && got; ++sp)
          got = wait_flag(flag(sp), ctl);
        if (!__all_sync(0xffffffffu, got)) break;
        // every flag of this warp is up (all lanes have acquired the partials):
        // lower them for the next launch (the launch boundary orders these
        // stores before that launch's raises)
        if (lane == 0)
          for (int sp = 0; sp < p.splits - 1; ++sp) ptx::st_relaxed_gpu(flag(sp), 0u);
        // fold the other splits' partials into this accumulator (fp32)
        for (int g = g0; g < g0 + kHalfG; ++g) {
          uint32_t v[4][8];
#pragma unroll
          for (int b = 0; b < 4; ++b) ptx::tmem_ld_32x32b_x8(gcol(g) + 32 * b, v[b]);
          ptx::tmem_wait_ld();
          for (int sp = 0; sp < p.splits - 1; ++sp) {
            const float4* src = part0 + static_cast<size_t>(sp) * CG * kSlotF4 + g * 256;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float4 a = __ldcg(src + 32 * k);
              v[0][k] = __float_as_uint(__uint_as_float(v[0][k]) + a.x);
              v[1][k] = __float_as_uint(__uint_as_float(v[1][k]) + a.y);
              v[2][k] = __float_as_uint(__uint_as_float(v[2][k]) + a.z);
              v[3][k] = __float_as_uint(__uint_as_float(v[3][k]) + a.w);
            }
          }
#pragma unroll
          for (int b = 0; b < 4; ++b) ptx::tmem_st_32x32b_x8(gcol(g) + 32 * b, v[b]);
        }
        ptx::tmem_wait_st();
      }
      // Column group g (32 output columns n0 + 32g + 4k + b, k < 8, b < 4) sits in
      // accumulator columns 128h + 32b + 8(g % 4) + k, h = g / 4; the quadrant's
      // other epilogue warp works on the other half of the groups.  First every
      // group of this warp is loaded, cleared, scaled and packed to 16 bits in
      // registers, and the accumulator goes back to the MMA issuers; only then
      // are the packed groups staged and stored (one 32-column TMA tile each),
      // while the next tile accumulates.
      // The first group goes straight to the staging tile (its previous store
      // finished reading long ago), the others are held in registers.
      constexpr int kRegG = kHalfG - 1;
      uint32_t pk[kRegG > 0 ? kRegG : 1][16];
      if (lane == 0) ptx::bulk_wait_group_read<0>();
      __syncwarp();
#pragma unroll
      for (int gl = 0; gl < kHalfG; ++gl) {
        const int g = g0 + gl;
        // two halves (accumulator columns 32b.., b = 2h, 2h + 1), so that only
        // 16 loaded registers are live next to the packed groups
        uint32_t v[16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t cur[2][8];
#pragma unroll
          for (int b = 0; b < 2; ++b)
            ptx::tmem_ld_32x32b_x8(gcol(g) + 32 * (2 * h + b), cur[b]);
          ptx::tmem_wait_ld();
          // read: clear these columns for the next tile's accumulation
#pragma unroll
          for (int b = 0; b < 2; ++b) ptx::tmem_st_32x32b_x8(gcol(g) + 32 * (2 * h + b), zero8);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            // columns 4k + 2h, 4k + 2h + 1 of the group
            const int o = 32 * gl + 4 * k + 2 * h;
            const float2 wc2 = *reinterpret_cast<const float2*>(wb + o);
            const float2 b2 = *reinterpret_cast<const float2*>(wb + BN / 2 + o);
            const float y0 = fmaf(__uint_as_float(cur[0][k]), wc2.x, b2.x);
            const float y1 = fmaf(__uint_as_float(cur[1][k]), wc2.y, b2.y);
            v[2 * k + h] = H::pack(y0, y1);
          }
        }
        if (gl == 0) {
          stage_row(stg, lane, v);
        } else {
#pragma unroll
          for (int x = 0; x < 16; ++x) pk[gl - 1][x] = v[x];
        }
      }
      // this warp's columns are read and cleared: release them to the MMA
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_remote(acc_empty0 + 8u * acc_stage);
#pragma unroll
      for (int gl = 0; gl < kHalfG; ++gl) {
        if (gl > 0) {
          // the staging tile must no longer be read by the previous store
          if (lane == 0) ptx::bulk_wait_group_read<0>();
          __syncwarp();
          stage_row(stg, lane, pk[gl - 1]);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          // staging row `lane` is output row m_cta + 4 * lane + q
          ptx::tma_store_3d(&tm_out, ptx::smem_u32(stg), n0 + 32 * (g0 + gl), m_cta / 4, q);
          ptx::bulk_commit_group();
        }
      }
    }
    if (lane == 0) ptx::bulk_wait_group<0>();
    __syncwarp();
  } else if (warp < 12) {
    // ------------------------------------------------------------ scale feeders
    // A unit's LoRA items come first, then its K-block items: two loops, so
    // the scale feed of the K-block items is compiled on its own.
    const int q = warp & 3;
    constexpr int kLuRowsF = L::kBNc / 8;  // LU' rows scaled per feeder warp
    int stage = 0;
    uint32_t phase = 0;
    const uint32_t full_bar0 = to_leader(full(0));
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    bool ok = true;
    for (int u = cluster_id; ok && u < p.num_units; u += num_clusters) {
      const Unit w = unit_of<SK>(p, u);
      const int t = w.tile;
      int mb, nb;
      tile_coords(p, t, mb, nb);
      const int m_cta = mb * kBM * CG + kBM * static_cast<int>(rank);
      const int n_cta = nb * BN + L::kBNc * static_cast<int>(rank);
      float lu_inv[(kLuRowsF + 31) / 32];
      for (int i = 0; i < w.lora; ++i) {
        if (!warp_wait_bar<false>(auxfull(stage), phase, kSiteSfAuxFull, ctl)) {
          ok = false;
          break;
        }
        // LoRA item: this warp builds LA' rows [32q, 32q + 32) (16-bit LA'
        // arrives ready) and scales its share of LU' (rows kBNc/2 + q kBNc/8 ..)
        int zero_col = -1, bad_col = -1;
        uint8_t* st = smem + stage * L::kStageBytes;
        if (!p.la16) {
          if (p.lora_tma)
            lora_la_from_smem<F16>(st + L::kLoraLA, st + L::kLoraRawLA, 32 * q, lane);
          else
            lora_la_direct<32, F16>(st + L::kLoraLA, p, m_cta, i, 32 * q, lane);
        }
        if ((p.lora_tma || p.la16) && p.wcscale != nullptr && !p.prepacked) {
          const int r0 = L::kBNc / 2 + q * kLuRowsF;
          if (p.la16)
            lora_lu_scale<kLuRowsF, 128, F16>(st + L::kLora16LU, st + L::kLoraWC, n_cta, p.N,
                                              r0, lane, i == 0, lu_inv, zero_col, bad_col);
          else
            lora_lu_scale<kLuRowsF, 64, F16>(st + L::kLoraLU, st + L::kLoraWC, n_cta, p.N, r0,
                                             lane, i == 0, lu_inv, zero_col, bad_col);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        // The pair peer's LoRA rows are generic shared-memory writes that the
        // leader's MMA reads: the proxy fence above orders them before this
        // arrival (CTA-scope release, as for every other arrival here).
        if (lane == 0) ptx::mbar_arrive_remote(full_bar0 + 8u * stage);
        // LoRA operands the accumulator cannot carry (this warp's LU' rows),
        // reported after the arrival
        warp_report_lora(p.status, kStatusWcscaleZero, zero_col >= 0, zero_col);
        warp_report_lora(p.status, kStatusLuOverflow, bad_col >= 0, bad_col);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // the K-block items, compiled once per scale layout
      auto feed_items = [&](auto packed_tag, auto act_tag) {
        constexpr bool kPacked = decltype(packed_tag)::value;
        constexpr bool kActPacked = decltype(act_tag)::value;
        for (int j = 0; ok && j < w.nkb; ++j) {
          if (!warp_wait_bar<false>(auxfull(stage), phase, kSiteSfAuxFull, ctl)) {
            ok = false;
            break;
          }
          const uint8_t* st = smem + stage * L::kStageBytes;
          // Every feeder writes the same words into its own lane quadrant:
          // the block-scaled MMA reads the scale words in every quadrant.
          const uint32_t col = tmem_base + lane_base +
                               static_cast<uint32_t>(L::kAccCols + stage * L::kSfCols);
          // Packed scales arrive as words [step][rows]: lane a's four words of a
          // 128-row block are 16 consecutive bytes (weights: prepacked;
          // activations: act_scales_packed).
#pragma unroll
          for (int kk = 0; kk < KBI; ++kk) {
            uint32_t a[16], b[16 * L::kSfbHalves];
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
              const int ks = 4 * kk + s4;
              if (kActPacked) {
                const uint4 va = lds128(st + L::kOffSFA + 4 * kBM * ks + 16 * lane);
                a[4 * s4] = va.x;
                a[4 * s4 + 1] = va.y;
                a[4 * s4 + 2] = va.z;
                a[4 * s4 + 3] = va.w;
              } else {
                sf_words(st + L::kOffSFA + 4 * kBM * ks, kBM, lane, a + 4 * s4);
              }
#pragma unroll
              for (int h = 0; h < L::kSfbHalves; ++h) {
                uint32_t* bw = b + 4 * (s4 * L::kSfbHalves + h);
                if (kPacked) {
                  const uint4 v =
                      lds128(st + L::kOffSFB + 4 * BN * ks + 4 * (128 * h + 4 * lane));
                  bw[0] = v.x;
                  bw[1] = v.y;
                  bw[2] = v.z;
                  bw[3] = v.w;
                } else {
                  sf_words(st + L::kOffSFB + 4 * BN * ks + 128 * h, BN, lane, bw);
                }
              }
            }
            if (KBI == 1 && L::kSfbHalves == 2) {
              // one K block: SFA (16 columns) and SFB (32) are adjacent; two
              // stores instead of three (each store briefly holds up the MMAs)
              uint32_t v[32];
#pragma unroll
              for (int x = 0; x < 16; ++x) {
                v[x] = a[x];
                v[16 + x] = b[x];
              }
              ptx::tmem_st_32x32b_x32(col, v);
              ptx::tmem_st_32x32b_x16(col + 32, b + 16);
            } else {
              ptx::tmem_st_32x32b_x16(col + 16 * kk, a);
#pragma unroll
              for (int h = 0; h < L::kSfbHalves; ++h)
                ptx::tmem_st_32x32b_x16(col + 4 * L::kSteps + 16 * L::kSfbHalves * kk + 16 * h,
                                        b + 16 * h);
            }
          }
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive_remote(full_bar0 + 8u * stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      };
      if (p.prepacked) {
        if (p.act_packed)
          feed_items(std::true_type{}, std::true_type{});
        else
          feed_items(std::true_type{}, std::false_type{});
      } else if (p.act_packed) {
        feed_items(std::false_type{}, std::true_type{});
      } else {
        feed_items(std::false_type{}, std::false_type{});
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (CG == 2) ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    if (CG == 2)
      ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace svdq
