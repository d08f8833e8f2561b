// svdq_api.cu -- the C ABI declared in include/svdq.h: argument validation,
// the launch planner (tile choice, shared-memory pipeline-depth solver,
// tensor-memory column budget, persistent grid), TMA tensor-map encoding and
// the kernel launch.  Host code only touches the device through the CUDA
// runtime; nothing here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "svdq.h"
#include "svdq_kernel.cuh"
#include "svdq_prepack.cuh"
#include "svdq_quant.cuh"

namespace svdq {

// Device status word: [0] code, [1] wait site, [2] CTA, [3] spare.
__device__ int g_device_status[4];

// Scratch of svdq_w4a4_gemm_split_noalloc, for callers that cannot allocate
// device memory.  Every GPU that loads this library holds it (zero-filled at
// load) until the process exits; only that entry point touches it.
static __device__ __align__(256) uint8_t g_noalloc_scratch[SVDQ_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kGb300SmemOptin = 232448;  // 227 KB dynamic shared memory per block
constexpr int kMaxDevices = 64;
constexpr int kDefaultTimeoutMs = 2000;
constexpr int kMaxSplits = 8;
constexpr int kMinSplitBlocks = 8;  // planner's minimum K blocks per split
constexpr int64_t kWsAlign = 256;

struct DeviceInfo {
  bool probed = false;
  bool supported = false;
  int sm_count = 0;
  int smem_optin = 0;
  int* status = nullptr;
  void* noalloc_scratch = nullptr;  // device address of g_noalloc_scratch, looked up once
  // per kernel: (1,128), (1,256), (2,256) with bf16 I/O, the same with fp16,
  // then those six with split-K
  bool attr_set[12] = {};
  int max_clusters[12] = {};
  int quant_smem_set[2] = {};  // activation quantiser (bf16, fp16): opted-in smem bytes
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

struct Plan {
  int cta_group = 1;
  int tile_n = 0;
  int stages = 0;
  int acc_stages = 0;
  int stage_bytes = 0;
  int lora_block_bytes = 0;
  int lora_blocks = 0;
  int k_blocks = 0;
  int main_items = 0;
  int kbi = 1;
  int r16 = 0;
  int smem_bytes = 0;
  int tmem_cols_used = 0;
  int tiles_m = 0, tiles_n = 0;
  long long num_tiles = 0;
  int splits = 1;
  long long num_units = 0;
  int64_t ws_partial_bytes = 0, ws_flag_bytes = 0;
  int grid = 0;  // CTAs
  int sm_count = 0;
  int group_m = 0;
};

int validate_options(const svdq_options_t* o) {
  if (o == nullptr) return SVDQ_OK;
  if (o->tile_n != 0 && o->tile_n != 128 && o->tile_n != 256) return SVDQ_ERR_BAD_OPTION;
  if (o->stages != 0 && (o->stages < 2 || o->stages > kMaxStages)) return SVDQ_ERR_BAD_OPTION;
  if (o->max_ctas < 0 || o->timeout_ms < 0) return SVDQ_ERR_BAD_OPTION;
  if (o->debug_fault != 0 && o->debug_fault != 1) return SVDQ_ERR_BAD_OPTION;
  if (o->cta_group < 0 || o->cta_group > 2) return SVDQ_ERR_BAD_OPTION;
  if (o->cta_group == 2 && o->tile_n == 128) return SVDQ_ERR_BAD_OPTION;
  if (o->io_dtype != SVDQ_IO_BF16 && o->io_dtype != SVDQ_IO_FP16) return SVDQ_ERR_BAD_OPTION;
  if (o->k_splits < -1 || o->k_splits > kMaxSplits) return SVDQ_ERR_BAD_OPTION;
  if (o->act_scales_packed != 0 && o->act_scales_packed != 1) return SVDQ_ERR_BAD_OPTION;
  if (o->relaxed_order != 0 && o->relaxed_order != 1) return SVDQ_ERR_BAD_OPTION;
  if (o->lora_act_16bit != 0 && o->lora_act_16bit != 1) return SVDQ_ERR_BAD_OPTION;
  return SVDQ_OK;
}

int validate_shape(int64_t M, int64_t N, int64_t K, int64_t R) {
  if (M < 0 || N < 0 || K <= 0 || R < 0) return SVDQ_ERR_INVALID_ARG;
  if (M % 16 || N % 16 || K % 64) return SVDQ_ERR_UNSUPPORTED_SHAPE;
  if (M > SVDQ_MAX_MN || N > SVDQ_MAX_MN || K > SVDQ_MAX_K || R > SVDQ_MAX_RANK)
    return SVDQ_ERR_UNSUPPORTED_SHAPE;
  return SVDQ_OK;
}

// Per-(CTA group, tile) constants the solver needs.
struct TileInfo {
  int stage_bytes, acc_cols, sf_cols, acc_stages, fixed_smem, lora_block_bytes, kbi;
};

// K blocks per main ring item.  One: five single-block stages keep more
// loads in flight than two double-block stages, and the MMA issuer's per-item
// cost (one barrier wait, one commit) stays below four K=64 MMAs.
template <int CG>
constexpr int kbi_for() {
  return 1;
}

template <int CG, int BN>
TileInfo tile_info() {
  using L = Layout<CG, BN, kbi_for<CG>()>;
  // LoRA ring item: LA' [128][32] bf16 + LU' [BN/CG][32] bf16 + raw LA [128][32] fp32
  // + wcscale; all inside one stage (both operands divided across a pair).
  return TileInfo{L::kStageBytes, L::kAccCols, L::kSfCols, L::kAccStages, L::smem_bytes(0),
                  kBM * kLoraRanks * 2 + L::kBNc * kLoraRanks * 2 + kBM * kLoraRanks * 4 +
                      2 * L::kBNc,
                  L::kKbi};
}

TileInfo tile_info_for(int cg, int bn) {
  if (cg == 2) return tile_info<2, 256>();
  return bn == 256 ? tile_info<1, 256>() : tile_info<1, 128>();
}

// Tile choice.  Candidates: a CTA pair with a 256 x 256 cluster tile (each CTA
// streams half the operand bytes per MMA), single CTAs with 128 x 256 or
// 128 x 128 tiles.  Unless the caller forces one, the candidate with the least
// estimated time wins: waves x per-SM tile work / relative efficiency, where
// waves = ceil(tiles / (SMs / cg)) and the efficiencies (1, 0.87, 0.75) are the
// measured large-shape throughputs relative to the pair.  A pair needs at
// least 256 rows and columns (below that half its work would be padding).
void choose_tile(int64_t M, int64_t N, const svdq_options_t* o, int sm_count, int* cg, int* bn) {
  const int fc = (o && o->cta_group) ? o->cta_group : 0;
  const int fn = (o && o->tile_n) ? o->tile_n : 0;
  struct Cand {
    int cg, bn;
    double eff;
  };
  const Cand cands[3] = {{2, 256, 1.0}, {1, 256, 0.87}, {1, 128, 0.75}};
  const int sms = sm_count > 0 ? sm_count : 1;
  double best = 0.0;
  int bc = 0, bb = 0;
  for (const Cand& c : cands) {
    if (fc && c.cg != fc) continue;
    if (fn && c.bn != fn) continue;
    if (c.cg == 2 && !fc && (M < 256 || N < 256)) continue;
    const int64_t tiles = ((M + 128 * c.cg - 1) / (128 * c.cg)) * ((N + c.bn - 1) / c.bn);
    const int64_t units = sms / c.cg > 0 ? sms / c.cg : 1;
    const int64_t waves = (tiles + units - 1) / units;
    const double cost = static_cast<double>(waves) * 128.0 * c.bn / c.eff;
    if (bc == 0 || cost < best) {
      best = cost;
      bc = c.cg;
      bb = c.bn;
    }
  }
  if (bc == 0) {  // a forced combination outside the table (rejected later)
    bc = fc ? fc : 1;
    bb = fn ? fn : 256;
  }
  *cg = bc;
  *bn = bb;
}

// K splits (split-K), for launches whose tiles leave more than half of the
// clusters idle.  Every unit gets a cluster of its own (units <= clusters that
// fit at once), so all units of a tile run concurrently and the final split's
// wait for the other splits' partials always ends.  A split costs about as
// much as ten K blocks of MMA work (partial store, flag, fold), so the planner
// keeps at least kMinSplitBlocks K blocks per split: long-K shapes only.
// `allow` is false for entry points without a workspace.
int choose_splits(const Plan& pl, const svdq_options_t* o, long long avail, bool allow,
                  int* splits) {
  const int ks = o ? o->k_splits : 0;
  *splits = 1;
  if (ks >= 2) {
    if (!allow) return SVDQ_ERR_WORKSPACE;
    if (ks > pl.main_items || pl.num_tiles * ks > avail) return SVDQ_ERR_BAD_OPTION;
    *splits = ks;
  } else if (allow && ks != 1 && pl.num_tiles * 2 <= avail) {
    long long sp = avail / pl.num_tiles;
    if (sp > pl.main_items / kMinSplitBlocks) sp = pl.main_items / kMinSplitBlocks;
    if (sp > kMaxSplits) sp = kMaxSplits;
    if (sp >= 2) *splits = static_cast<int>(sp);
  }
  return SVDQ_OK;
}

int make_plan(int64_t M, int64_t N, int64_t K, int64_t R, const svdq_options_t* o, int sm_count,
              int smem_optin, int max_clusters, Plan* out, bool allow_split) {
  Plan pl;
  choose_tile(M, N, o, sm_count, &pl.cta_group, &pl.tile_n);
  const TileInfo ti = tile_info_for(pl.cta_group, pl.tile_n);
  // Pipeline depth: whatever shared memory is left after the epilogue staging,
  // per-warp wcscale/bias and barriers, capped by the tensor-memory columns
  // left after the accumulators.  LoRA needs no dedicated buffer: its ring
  // items reuse main stages.
  const int by_smem = (smem_optin - ti.fixed_smem) / ti.stage_bytes;
  const int by_tmem = (kTmemCols - ti.acc_cols) / ti.sf_cols;
  int max_stages = by_smem < by_tmem ? by_smem : by_tmem;
  if (max_stages > kMaxStages) max_stages = kMaxStages;
  if (o && o->stages) {
    if (o->stages > max_stages) return SVDQ_ERR_BAD_OPTION;
    pl.stages = o->stages;
  } else {
    pl.stages = max_stages;
  }
  if (pl.stages < 2) return SVDQ_ERR_UNSUPPORTED_DEVICE;
  pl.stage_bytes = ti.stage_bytes;
  pl.acc_stages = ti.acc_stages;
  pl.smem_bytes = ti.fixed_smem + pl.stages * ti.stage_bytes;
  pl.tmem_cols_used = ti.acc_cols + pl.stages * ti.sf_cols;
  // 16-bit LA': 64-rank items of LA' [128][64] + LU' [tile_n / cg][64] + wcscale
  const bool la16 = o && o->lora_act_16bit;
  const int lora_ranks = la16 ? 64 : kLoraRanks;
  pl.lora_block_bytes =
      la16 ? kBM * 128 + (pl.tile_n / pl.cta_group) * 130 : ti.lora_block_bytes;
  pl.k_blocks = static_cast<int>((K + kBK - 1) / kBK);
  pl.kbi = ti.kbi;
  pl.main_items = (pl.k_blocks + pl.kbi - 1) / pl.kbi;
  pl.lora_blocks = static_cast<int>((R + lora_ranks - 1) / lora_ranks);
  pl.r16 = static_cast<int>((R + 15) / 16 * 16);
  const int tm = kBM * pl.cta_group;
  pl.tiles_m = static_cast<int>((M + tm - 1) / tm);
  pl.tiles_n = static_cast<int>((N + pl.tile_n - 1) / pl.tile_n);
  pl.num_tiles = static_cast<long long>(pl.tiles_m) * pl.tiles_n;
  if (pl.num_tiles >= (1LL << 31)) return SVDQ_ERR_UNSUPPORTED_SHAPE;
  pl.sm_count = sm_count;
  long long clusters = sm_count / pl.cta_group;
  if (max_clusters > 0 && clusters > max_clusters) clusters = max_clusters;
  if (o && o->max_ctas > 0 && clusters * pl.cta_group > o->max_ctas)
    clusters = o->max_ctas / pl.cta_group > 0 ? o->max_ctas / pl.cta_group : 1;
  int rc = choose_splits(pl, o, clusters, allow_split, &pl.splits);
  if (rc != SVDQ_OK) return rc;
  pl.num_units = pl.num_tiles * pl.splits;
  if (clusters > pl.num_units) clusters = pl.num_units;
  // Balanced persistent grid: keep the number of rounds (units per cluster on
  // the busiest cluster) and use the fewest clusters that need no more, so every
  // cluster gets the same number of units, give or take one (192 tiles on 76
  // pairs: 3 rounds -> 64 pairs).  Less contention for the same critical path.
  if (clusters > 0) {
    const long long rounds = (pl.num_units + clusters - 1) / clusters;
    clusters = (pl.num_units + rounds - 1) / rounds;
  }
  pl.grid = static_cast<int>(clusters * pl.cta_group);
  if (pl.splits > 1) {
    // fp32 partial tiles of the non-final splits (one slot per tile, split,
    // CTA), then one flag per slot and epilogue warp (eight per CTA)
    const int64_t slots = static_cast<int64_t>(pl.num_tiles) * (pl.splits - 1) * pl.cta_group;
    pl.ws_partial_bytes = slots * kBM * pl.tile_n * 4;
    pl.ws_flag_bytes = slots * 8 * 4;
  }
  pl.group_m = pl.tiles_m < 8 ? (pl.tiles_m > 0 ? pl.tiles_m : 1) : 8;
  *out = pl;
  return SVDQ_OK;
}

int probe_device(int* dev_out, DeviceInfo** info_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SVDQ_ERR_UNSUPPORTED_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return SVDQ_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& d = g_devices[dev];
  if (!d.probed) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess) {
      cudaGetLastError();
      return SVDQ_ERR_UNSUPPORTED_DEVICE;
    }
    d.supported = (major == 10 && minor == 3);
    if (d.supported) {
      void* sym = nullptr;
      if (cudaGetSymbolAddress(&sym, g_device_status) != cudaSuccess) {
        cudaGetLastError();
        return SVDQ_ERR_CUDA;
      }
      d.status = static_cast<int*>(sym);
      if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr) {
          cudaGetLastError();
          return SVDQ_ERR_CUDA;
        }
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      }
    }
    d.probed = true;
  }
  if (!d.supported) return SVDQ_ERR_UNSUPPORTED_DEVICE;
  *dev_out = dev;
  *info_out = &d;
  return SVDQ_OK;
}

constexpr int kernel_index(int cg, int bn, bool f16, bool sk) {
  return (cg == 2 ? 2 : (bn == 256 ? 1 : 0)) + (f16 ? 3 : 0) + (sk ? 6 : 0);
}

// Once per device and kernel: opt in to the shared memory and find how many
// clusters fit at once.
template <int CG, int BN, bool F16, bool SK>
int ensure_kernel(DeviceInfo* d, int smem_bytes) {
  std::lock_guard<std::mutex> lock(g_mutex);
  const int idx = kernel_index(CG, BN, F16, SK);
  if (!d->attr_set[idx]) {
    auto k = svdq_w4a4_kernel<CG, BN, kbi_for<CG>(), F16, SK>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, d->smem_optin) !=
        cudaSuccess) {
      cudaGetLastError();
      return SVDQ_ERR_CUDA;
    }
    d->max_clusters[idx] = d->sm_count / CG;
    if (CG == 2) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * (d->sm_count / 2));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = smem_bytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) == cudaSuccess && n > 0)
        d->max_clusters[idx] = n;
      cudaGetLastError();
    }
    d->attr_set[idx] = true;
  }
  return SVDQ_OK;
}

// rank 1..3; strides_bytes holds rank - 1 strides (dimensions 1..rank-1).
int encode(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
           const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
           CUtensorMapSwizzle swz) {
  cuuint64_t gd[3] = {1, 1, 1};
  cuuint64_t gs[2] = {0, 0};
  cuuint32_t bx[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    if (i > 0) gs[i - 1] = strides_bytes[i - 1];
  }
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r =
      g_encode(map, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gd, gs, bx, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SVDQ_OK : SVDQ_ERR_CUDA;
}

struct Operands {
  const void *act, *wgt, *ascales, *wscales, *la, *lu, *wc, *bias;
  void* out;
};

template <int CG, int BN, bool F16, bool SK>
int launch(const Plan& pl, DeviceInfo* dinfo, const Operands& op, const KParams& kp, int64_t M,
           int64_t N, int64_t K, int64_t R, cudaStream_t stream) {
  constexpr int KBI = kbi_for<CG>();
  using L = Layout<CG, BN, KBI>;
  constexpr CUtensorMapDataType kIoType =
      F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  (void)dinfo;
  int rc = SVDQ_OK;
  alignas(64) CUtensorMap tm[8];
  const uint64_t u = static_cast<uint64_t>(K / 2);
  // Row-quad views of row-major [rows][width] operands: dims (width, rows / 4,
  // 4) with strides (4 rows, 1 row).  A box (w, 32, 4) lands in shared memory
  // as 128 rows in which row a + 32b is matrix row 4a + b of the block.
  const uint64_t M4 = static_cast<uint64_t>(M / 4), N4 = static_cast<uint64_t>(N / 4);
  {
    const uint64_t d_act[3] = {u, M4, 4}, s_act[2] = {4 * u, u};
    const uint32_t b_quad[3] = {128, 32, 4};
    if ((rc = encode(&tm[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, op.act, d_act, s_act, b_quad,
                     CU_TENSOR_MAP_SWIZZLE_128B)) != SVDQ_OK)
      return rc;
    const uint64_t d_wgt[3] = {u, N4, 4};
    if ((rc = encode(&tm[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, op.wgt, d_wgt, s_act, b_quad,
                     CU_TENSOR_MAP_SWIZZLE_128B)) != SVDQ_OK)
      return rc;
    if (kp.act_packed) {
      // packed activation scale words uint32 [K/64][M]: 16 * kBM bytes per K block
      const uint64_t d_sfa[2] = {static_cast<uint64_t>(M), static_cast<uint64_t>(K / 64)},
                     s_sfa[1] = {static_cast<uint64_t>(M) * 4};
      const uint32_t b_sfa[2] = {kBM, 4 * KBI};
      if ((rc = encode(&tm[2], CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, op.ascales, d_sfa, s_sfa,
                       b_sfa, CU_TENSOR_MAP_SWIZZLE_NONE)) != SVDQ_OK)
        return rc;
    } else {
      const uint64_t d_sfa[2] = {static_cast<uint64_t>(M), static_cast<uint64_t>(K / 16)},
                     s_sfa[1] = {static_cast<uint64_t>(M)};
      const uint32_t b_sfa[2] = {kBM, 16 * KBI};
      if ((rc = encode(&tm[2], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, op.ascales, d_sfa, s_sfa, b_sfa,
                       CU_TENSOR_MAP_SWIZZLE_NONE)) != SVDQ_OK)
        return rc;
    }
    if (kp.prepacked) {
      // packed scale words uint32 [K/64][N]: the same 16 * BN bytes per K block
      const uint64_t d_sfb[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K / 64)},
                     s_sfb[1] = {static_cast<uint64_t>(N) * 4};
      const uint32_t b_sfb[2] = {BN, 4 * KBI};
      if ((rc = encode(&tm[3], CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, op.wscales, d_sfb, s_sfb,
                       b_sfb, CU_TENSOR_MAP_SWIZZLE_NONE)) != SVDQ_OK)
        return rc;
    } else {
      const uint64_t d_sfb[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K / 16)},
                     s_sfb[1] = {static_cast<uint64_t>(N)};
      const uint32_t b_sfb[2] = {BN, 16 * KBI};
      if ((rc = encode(&tm[3], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, op.wscales, d_sfb, s_sfb, b_sfb,
                       CU_TENSOR_MAP_SWIZZLE_NONE)) != SVDQ_OK)
        return rc;
    }
    // output: one store writes 32 columns of rows 4a + q (a < 32) of a 128-row block
    const uint64_t d_out[3] = {static_cast<uint64_t>(N), M4, 4},
                   s_out[2] = {static_cast<uint64_t>(N) * 8, static_cast<uint64_t>(N) * 2};
    const uint32_t b_out[3] = {32, 32, 1};
    if ((rc = encode(&tm[7], kIoType, 3, op.out, d_out, s_out, b_out,
                     CU_TENSOR_MAP_SWIZZLE_64B)) != SVDQ_OK)
      return rc;
  }
  if (kp.la16) {
    // 16-bit LA' and LU: 64 ranks (128 bytes) per box, 128-byte swizzle,
    // row-quad order like the operand tiles
    const uint64_t r64 = static_cast<uint64_t>(R);
    const uint64_t d_la[3] = {r64, M4, 4}, s_la[2] = {8 * r64, 2 * r64};
    const uint32_t b_lora[3] = {64, 32, 4};
    if ((rc = encode(&tm[4], kIoType, 3, op.la, d_la, s_la, b_lora,
                     CU_TENSOR_MAP_SWIZZLE_128B)) != SVDQ_OK)
      return rc;
    const uint64_t d_lu[3] = {r64, N4, 4};
    if ((rc = encode(&tm[5], kIoType, 3, op.lu, d_lu, s_la, b_lora,
                     CU_TENSOR_MAP_SWIZZLE_128B)) != SVDQ_OK)
      return rc;
  } else if (kp.lora_tma) {
    const uint64_t r64 = static_cast<uint64_t>(R);
    const uint64_t d_la[3] = {r64, M4, 4}, s_la[2] = {16 * r64, 4 * r64};
    const uint32_t b_lora[3] = {kLoraRanks, 32, 4};
    if ((rc = encode(&tm[4], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, op.la, d_la, s_la, b_lora,
                     CU_TENSOR_MAP_SWIZZLE_NONE)) != SVDQ_OK)
      return rc;
    const uint64_t d_lu[3] = {r64, N4, 4}, s_lu[2] = {8 * r64, 2 * r64};
    if ((rc = encode(&tm[5], kIoType, 3, op.lu, d_lu, s_lu, b_lora,
                     CU_TENSOR_MAP_SWIZZLE_64B)) != SVDQ_OK)
      return rc;
  } else {
    tm[4] = tm[0];  // unused
    tm[5] = tm[0];
  }
  if (op.wc != nullptr) {
    const uint64_t d_wc[1] = {static_cast<uint64_t>(N)};
    const uint32_t b_wc[1] = {L::kBNc};
    if ((rc = encode(&tm[6], kIoType, 1, op.wc, d_wc, nullptr, b_wc,
                     CU_TENSOR_MAP_SWIZZLE_NONE)) != SVDQ_OK)
      return rc;
  } else {
    tm[6] = tm[0];  // unused
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  // the kernel waits (griddepcontrol.wait) before touching memory, so it may
  // be scheduled while the previous kernel in the stream finishes
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CG;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CG == 2 ? 2 : 1;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, svdq_w4a4_kernel<CG, BN, KBI, F16, SK>, tm[0], tm[1], tm[2],
                         tm[3], tm[4], tm[5], tm[6], tm[7], kp);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return SVDQ_ERR_LAUNCH;
  }
  return SVDQ_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Runtime (CTA group, tile, I/O type, split-K) -> kernel instance.
int ensure_any(int cg, int bn, bool f16, bool sk, DeviceInfo* d) {
  const int so = d->smem_optin;
  if (sk) {
    if (cg == 2)
      return f16 ? ensure_kernel<2, 256, true, true>(d, so)
                 : ensure_kernel<2, 256, false, true>(d, so);
    if (bn == 256)
      return f16 ? ensure_kernel<1, 256, true, true>(d, so)
                 : ensure_kernel<1, 256, false, true>(d, so);
    return f16 ? ensure_kernel<1, 128, true, true>(d, so)
               : ensure_kernel<1, 128, false, true>(d, so);
  }
  if (cg == 2)
    return f16 ? ensure_kernel<2, 256, true, false>(d, so)
               : ensure_kernel<2, 256, false, false>(d, so);
  if (bn == 256)
    return f16 ? ensure_kernel<1, 256, true, false>(d, so)
               : ensure_kernel<1, 256, false, false>(d, so);
  return f16 ? ensure_kernel<1, 128, true, false>(d, so)
             : ensure_kernel<1, 128, false, false>(d, so);
}

template <bool F16, bool SK>
int launch_any(const Plan& pl, DeviceInfo* dinfo, const Operands& op, const KParams& kp, int64_t M,
               int64_t N, int64_t K, int64_t R, cudaStream_t s) {
  if (pl.cta_group == 2) return launch<2, 256, F16, SK>(pl, dinfo, op, kp, M, N, K, R, s);
  if (pl.tile_n == 256) return launch<1, 256, F16, SK>(pl, dinfo, op, kp, M, N, K, R, s);
  return launch<1, 128, F16, SK>(pl, dinfo, op, kp, M, N, K, R, s);
}

// The plan a launch on this device uses: tile choice, the kernel's
// attributes and co-resident cluster count, then the solver.
int device_plan(int64_t M, int64_t N, int64_t K, int64_t R, const svdq_options_t* options,
                DeviceInfo* dinfo, bool f16, bool allow_split, Plan* pl) {
  int cg = 1, bn = 256;
  choose_tile(M, N, options, dinfo->sm_count, &cg, &bn);
  // the unsplit instance's co-resident clusters (the split instance has the
  // same shared memory and threads)
  int rc = ensure_any(cg, bn, f16, false, dinfo);
  if (rc != SVDQ_OK) return rc;
  const int idx = kernel_index(cg, bn, f16, false);
  if ((rc = make_plan(M, N, K, R, options, dinfo->sm_count, dinfo->smem_optin,
                      dinfo->max_clusters[idx], pl, allow_split)) != SVDQ_OK)
    return rc;
  return pl->splits > 1 ? ensure_any(cg, bn, f16, true, dinfo) : SVDQ_OK;
}

int64_t ws_flag_offset(const Plan& pl) {
  return (pl.ws_partial_bytes + kWsAlign - 1) / kWsAlign * kWsAlign;
}
int64_t ws_bytes(const Plan& pl) {
  return pl.splits > 1 ? ws_flag_offset(pl) + pl.ws_flag_bytes : 0;
}

// One operator call; `prepacked` selects packed scale words and LU' (from
// svdq_prepack_weights) for wscales / lora_up; a non-null workspace allows
// split-K.
int run_gemm(const void* act, const void* wgt, const void* ascales, const void* wscales,
             const float* lora_act_in, const void* lora_up, const void* wcscale, const void* bias,
             void* out, int64_t M, int64_t N, int64_t K, int64_t R, const svdq_options_t* options,
             void* stream, bool prepacked, void* workspace, int64_t workspace_bytes) {
  int rc = validate_options(options);
  if (rc != SVDQ_OK) return rc;
  const bool f16 = options != nullptr && options->io_dtype == SVDQ_IO_FP16;
  if (!act || !wgt || !ascales || !wscales || !out) return SVDQ_ERR_INVALID_ARG;
  if (R > 0 && (!lora_act_in || !lora_up)) return SVDQ_ERR_INVALID_ARG;
  if ((rc = validate_shape(M, N, K, R)) != SVDQ_OK) return rc;
  const bool la16 = options != nullptr && options->lora_act_16bit && R > 0;
  // 16-bit LA' rows go through TMA: their stride (2R bytes) must be 16-byte aligned
  if (la16 && R % 8) return SVDQ_ERR_BAD_OPTION;
  const void* ptrs[] = {act, wgt, ascales, wscales, out, lora_act_in, lora_up, wcscale, bias};
  for (const void* p : ptrs)
    if (p && !aligned(p, 16)) return SVDQ_ERR_MISALIGNED;
  if (M == 0 || N == 0) return SVDQ_OK;

  int dev = 0;
  DeviceInfo* dinfo = nullptr;
  if ((rc = probe_device(&dev, &dinfo)) != SVDQ_OK) return rc;
  Plan pl;
  if ((rc = device_plan(M, N, K, R, options, dinfo, f16, workspace != nullptr, &pl)) != SVDQ_OK)
    return rc;

  KParams kp;
  std::memset(&kp, 0, sizeof kp);
  kp.M = static_cast<int>(M);
  kp.N = static_cast<int>(N);
  kp.K = static_cast<int>(K);
  kp.R = static_cast<int>(R);
  kp.tiles_m = pl.tiles_m;
  kp.tiles_n = pl.tiles_n;
  kp.num_tiles = static_cast<int>(pl.num_tiles);
  kp.group_m = pl.group_m;
  kp.k_blocks = pl.k_blocks;
  kp.main_items = pl.main_items;
  kp.lora_blocks = pl.lora_blocks;
  kp.r16 = pl.r16;
  kp.num_stages = pl.stages;
  kp.lora_tma = (R > 0 && R % 8 == 0);
  kp.la16 = la16 ? 1 : 0;
  kp.lora_ranks = la16 ? 64 : kLoraRanks;
  kp.prepacked = prepacked ? 1 : 0;
  kp.act_packed = (options != nullptr && options->act_scales_packed) ? 1 : 0;
  kp.splits = pl.splits;
  kp.num_units = static_cast<int>(pl.num_units);
  if (pl.splits > 1) {
    if (!aligned(workspace, kWsAlign) || workspace_bytes < ws_bytes(pl)) return SVDQ_ERR_WORKSPACE;
    kp.partials = static_cast<float4*>(workspace);
    kp.flags =
        reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(workspace) + ws_flag_offset(pl));
  }
  kp.debug_fault = options ? options->debug_fault : 0;
  kp.ordered = (options != nullptr && options->relaxed_order) ? 0 : 1;
  const int tmo = (options && options->timeout_ms) ? options->timeout_ms : kDefaultTimeoutMs;
  kp.timeout_ns = static_cast<unsigned long long>(tmo) * 1000000ull;
  kp.lora_act_in = R > 0 ? lora_act_in : nullptr;
  kp.lora_up = R > 0 ? static_cast<const uint16_t*>(lora_up) : nullptr;
  kp.wcscale = static_cast<const uint16_t*>(wcscale);
  kp.bias = static_cast<const uint16_t*>(bias);
  kp.status = dinfo->status;

  const Operands op{act, wgt, ascales, wscales, lora_act_in, lora_up, wcscale, bias, out};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool sk = pl.splits > 1;
  if (f16)
    return sk ? launch_any<true, true>(pl, dinfo, op, kp, M, N, K, R, s)
              : launch_any<true, false>(pl, dinfo, op, kp, M, N, K, R, s);
  return sk ? launch_any<false, true>(pl, dinfo, op, kp, M, N, K, R, s)
            : launch_any<false, false>(pl, dinfo, op, kp, M, N, K, R, s);
}


// ---------------------------------------------------------------- activation quantiser
struct QuantPlan {
  int tiles = 0, splits = 1, stages = 0, r16 = 0, tmem_cols = 0, smem = 0, chunks = 0;
};

// One CTA per 128-row tile and K range.  A row tile is split along K over a
// cluster of 2, 4 or 8 CTAs while the tiles alone would leave SMs idle (each
// CTA streams its own part of x; the LoRA-down partials are added inside the
// cluster).  Ring depth: as many 64-wide K chunks as fit, up to ten: a chunk's
// round trip (HBM latency under load, then the quantisers) is about 2.5 us,
// and covering it at 50 GB/s per SM takes well over 100 KB in flight.
int plan_quant(int64_t M, int64_t K, int64_t R, int sm_count, int smem_optin, QuantPlan* q) {
  q->tiles = static_cast<int>((M + kQRows - 1) / kQRows);
  q->chunks = static_cast<int>(K / kQChunk);
  q->splits = 1;
  while (2 * q->splits <= kQMaxSplits && 2 * q->splits <= q->chunks &&
         static_cast<long long>(q->tiles) * 2 * q->splits <= sm_count)
    q->splits *= 2;
  q->r16 = R > 0 ? static_cast<int>((R + 15) / 16 * 16) : 0;
  q->tmem_cols = 0;
  if (q->r16 > 0) {
    q->tmem_cols = 32;
    while (q->tmem_cols < q->r16) q->tmem_cols *= 2;
  }
  const int room = smem_optin - quant_smem_bytes(q->r16, 0);
  q->stages = room / quant_stage_bytes(q->r16);
  if (q->stages > 10) q->stages = 10;
  if (q->stages < 3 || q->stages * quant_stage_bytes(q->r16) < quant_part_bytes(q->r16))
    return SVDQ_ERR_CUDA;
  q->smem = quant_smem_bytes(q->r16, q->stages);
  return SVDQ_OK;
}

template <bool F16>
int launch_quant(const QuantPlan& qp, DeviceInfo* dinfo, const void* x, const void* ld,
                 int64_t M, int64_t K, int64_t R, int packed, int la16, void* act, void* ascales,
                 void* la, cudaStream_t stream) {
  constexpr CUtensorMapDataType kIoType =
      F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  auto kern = svdq_quant_kernel<F16>;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    int& set = dinfo->quant_smem_set[F16 ? 1 : 0];
    if (set < qp.smem) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, qp.smem) !=
          cudaSuccess) {
        cudaGetLastError();
        return SVDQ_ERR_CUDA;
      }
      set = qp.smem;
    }
  }
  int rc = SVDQ_OK;
  alignas(64) CUtensorMap tm[2];
  // x [M][K] and lora_down [R][K]: 64-element (128-byte) boxes of 128 and R16
  // rows with the 128-byte swizzle the MMA descriptors expect
  const uint64_t d_x[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)},
                 s_x[1] = {static_cast<uint64_t>(K) * 2};
  const uint32_t b_x[2] = {kQChunk, kQRows};
  if ((rc = encode(&tm[0], kIoType, 2, x, d_x, s_x, b_x, CU_TENSOR_MAP_SWIZZLE_128B)) != SVDQ_OK)
    return rc;
  if (R > 0) {
    const uint64_t d_ld[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(R)};
    const uint32_t b_ld[2] = {kQChunk, static_cast<uint32_t>(qp.r16)};
    if ((rc = encode(&tm[1], kIoType, 2, ld, d_ld, s_x, b_ld, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        SVDQ_OK)
      return rc;
  } else {
    tm[1] = tm[0];  // unused
  }
  QParams p{};
  p.act = static_cast<uint8_t*>(act);
  p.ascales = static_cast<uint8_t*>(ascales);
  p.la = la;
  p.la16 = la16;
  p.M = static_cast<int>(M);
  p.K = static_cast<int>(K);
  p.R = static_cast<int>(R);
  p.r16 = qp.r16;
  p.chunks = qp.chunks;
  p.splits = qp.splits;
  p.stages = qp.stages;
  p.packed = packed;
  p.tmem_cols = qp.tmem_cols;
  p.status = dinfo->status;
  p.timeout_ns = static_cast<unsigned long long>(kDefaultTimeoutMs) * 1000000ull;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(qp.tiles * qp.splits));
  cfg.blockDim = dim3(kQThreads);
  cfg.dynamicSmemBytes = qp.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(qp.splits);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = qp.splits > 1 ? 2 : 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tm[0], tm[1], p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return SVDQ_ERR_LAUNCH;
  }
  return SVDQ_OK;
}

int validate_quant(const void* x, const void* ld, int64_t M, int64_t K, int64_t R,
                   int32_t io_dtype, int32_t packed, int32_t la16, const void* act,
                   const void* ascales, const void* la) {
  if (io_dtype != SVDQ_IO_BF16 && io_dtype != SVDQ_IO_FP16) return SVDQ_ERR_BAD_OPTION;
  if (packed != 0 && packed != 1) return SVDQ_ERR_BAD_OPTION;
  if (la16 != 0 && la16 != 1) return SVDQ_ERR_BAD_OPTION;
  if (M < 0 || K <= 0 || R < 0) return SVDQ_ERR_INVALID_ARG;
  if (M % 16 || K % 64 || M > SVDQ_MAX_MN || K > SVDQ_MAX_K || R > SVDQ_MAX_RANK)
    return SVDQ_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return SVDQ_OK;  // nothing to read or write (empty tensors may be NULL)
  if (!x || !act || !ascales) return SVDQ_ERR_INVALID_ARG;
  if ((R > 0) != (ld != nullptr) || (R > 0) != (la != nullptr)) return SVDQ_ERR_INVALID_ARG;
  const void* ptrs[] = {x, ld, act, ascales, la};
  for (const void* q : ptrs)
    if (q && !aligned(q, 16)) return SVDQ_ERR_MISALIGNED;
  return SVDQ_OK;
}

}  // namespace
}  // namespace svdq

using namespace svdq;

extern "C" int svdq_w4a4_gemm_ex(const void* act, const void* wgt, const void* ascales,
                                 const void* wscales, const float* lora_act_in,
                                 const void* lora_up, const void* wcscale, const void* bias,
                                 void* out, int64_t M, int64_t N, int64_t K, int64_t R,
                                 const svdq_options_t* options, void* stream) {
  return run_gemm(act, wgt, ascales, wscales, lora_act_in, lora_up, wcscale, bias, out, M, N, K,
                  R, options, stream, false, nullptr, 0);
}

extern "C" int svdq_w4a4_gemm_prepacked(const void* act, const void* wgt, const void* ascales,
                                        const void* wscales_packed, const float* lora_act_in,
                                        const void* lora_up_packed, const void* wcscale,
                                        const void* bias, void* out, int64_t M, int64_t N,
                                        int64_t K, int64_t R, const svdq_options_t* options,
                                        void* stream) {
  return run_gemm(act, wgt, ascales, wscales_packed, lora_act_in, lora_up_packed, wcscale, bias,
                  out, M, N, K, R, options, stream, true, nullptr, 0);
}

extern "C" int svdq_w4a4_gemm_split(const void* act, const void* wgt, const void* ascales,
                                    const void* wscales, const float* lora_act_in,
                                    const void* lora_up, const void* wcscale, const void* bias,
                                    void* out, int64_t M, int64_t N, int64_t K, int64_t R,
                                    const svdq_options_t* options, int32_t weights_prepacked,
                                    void* workspace, int64_t workspace_bytes, void* stream) {
  if (weights_prepacked != 0 && weights_prepacked != 1) return SVDQ_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < 0) return SVDQ_ERR_WORKSPACE;
  return run_gemm(act, wgt, ascales, wscales, lora_act_in, lora_up, wcscale, bias, out, M, N, K,
                  R, options, stream, weights_prepacked == 1, workspace, workspace_bytes);
}

extern "C" int64_t svdq_workspace_size(int64_t M, int64_t N, int64_t K, int64_t R,
                                       const svdq_options_t* options, int32_t sm_count) {
  int rc = validate_options(options);
  if (rc != SVDQ_OK) return rc;
  if ((rc = validate_shape(M, N, K, R)) != SVDQ_OK) return rc;
  if (M == 0 || N == 0) return 0;
  Plan pl;
  if (sm_count <= 0) {
    // exactly the plan a launch on the current device makes
    int dev = 0;
    DeviceInfo* d = nullptr;
    if ((rc = probe_device(&dev, &d)) != SVDQ_OK) return rc;
    const bool f16 = options != nullptr && options->io_dtype == SVDQ_IO_FP16;
    if ((rc = device_plan(M, N, K, R, options, d, f16, true, &pl)) != SVDQ_OK) return rc;
  } else if ((rc = make_plan(M, N, K, R, options, sm_count, kGb300SmemOptin, 0, &pl, true)) !=
             SVDQ_OK) {
    return rc;
  }
  return ws_bytes(pl);
}

extern "C" int svdq_pack_scales(const void* scales, int64_t rows, int64_t K, void* packed,
                                void* stream) {
  if (rows < 0 || K <= 0) return SVDQ_ERR_INVALID_ARG;
  if (rows % 16 || K % 64 || rows > SVDQ_MAX_MN || K > SVDQ_MAX_K)
    return SVDQ_ERR_UNSUPPORTED_SHAPE;
  if (!scales || !packed) return SVDQ_ERR_INVALID_ARG;
  if (!aligned(scales, 16) || !aligned(packed, 16)) return SVDQ_ERR_MISALIGNED;
  if (rows == 0) return SVDQ_OK;
  int dev = 0;
  DeviceInfo* dinfo = nullptr;
  int rc = probe_device(&dev, &dinfo);
  if (rc != SVDQ_OK) return rc;
  const long long work = (K / 64) * (rows / 4);
  long long blocks = (work + 255) / 256;
  const long long cap = 8LL * dinfo->sm_count;
  if (blocks > cap) blocks = cap;
  // the weight prepack kernel with no LoRA operand: its scale-word pass only
  svdq_prepack_kernel<false><<<static_cast<unsigned>(blocks), 256, 0,
                               static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t*>(scales), nullptr, nullptr, static_cast<uint32_t*>(packed),
      nullptr, static_cast<int>(rows), static_cast<int>(K), 0, dinfo->status);
  if (cudaGetLastError() != cudaSuccess) return SVDQ_ERR_LAUNCH;
  return SVDQ_OK;
}

extern "C" int svdq_prepack_weights(const void* wscales, const void* lora_up,
                                    const void* wcscale, int64_t N, int64_t K, int64_t R,
                                    int32_t io_dtype, void* wscales_packed,
                                    void* lora_up_packed, void* stream) {
  if (io_dtype != SVDQ_IO_BF16 && io_dtype != SVDQ_IO_FP16) return SVDQ_ERR_BAD_OPTION;
  if (N < 0 || K <= 0 || R < 0) return SVDQ_ERR_INVALID_ARG;
  if (N % 16 || K % 64 || N > SVDQ_MAX_MN || K > SVDQ_MAX_K || R > SVDQ_MAX_RANK)
    return SVDQ_ERR_UNSUPPORTED_SHAPE;
  if (!wscales || !wscales_packed) return SVDQ_ERR_INVALID_ARG;
  if (R > 0 && (!lora_up || !lora_up_packed)) return SVDQ_ERR_INVALID_ARG;
  const void* ptrs[] = {wscales, wscales_packed, lora_up, lora_up_packed, wcscale};
  for (const void* p : ptrs)
    if (p && !aligned(p, 16)) return SVDQ_ERR_MISALIGNED;
  if (N == 0) return SVDQ_OK;
  int dev = 0;
  DeviceInfo* dinfo = nullptr;
  int rc = probe_device(&dev, &dinfo);
  if (rc != SVDQ_OK) return rc;
  const long long work = (K / 64) * (N / 4) + N * R;
  long long blocks = (work + 255) / 256;
  const long long cap = 8LL * dinfo->sm_count;
  if (blocks > cap) blocks = cap;
  const uint8_t* ws = static_cast<const uint8_t*>(wscales);
  const uint16_t* lu = R > 0 ? static_cast<const uint16_t*>(lora_up) : nullptr;
  const uint16_t* wc = static_cast<const uint16_t*>(wcscale);
  uint32_t* wpk = static_cast<uint32_t*>(wscales_packed);
  uint16_t* lup = R > 0 ? static_cast<uint16_t*>(lora_up_packed) : nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int n = static_cast<int>(N), k = static_cast<int>(K), r = static_cast<int>(R);
  if (io_dtype == SVDQ_IO_FP16)
    svdq_prepack_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        ws, lu, wc, wpk, lup, n, k, r, dinfo->status);
  else
    svdq_prepack_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        ws, lu, wc, wpk, lup, n, k, r, dinfo->status);
  if (cudaGetLastError() != cudaSuccess) return SVDQ_ERR_LAUNCH;
  return SVDQ_OK;
}

extern "C" int svdq_w4a4_gemm(const void* act, const void* wgt, const void* ascales,
                              const void* wscales, const float* lora_act_in, const void* lora_up,
                              const void* wcscale, const void* bias, void* out, int64_t M,
                              int64_t N, int64_t K, int64_t R, void* stream) {
  return svdq_w4a4_gemm_ex(act, wgt, ascales, wscales, lora_act_in, lora_up, wcscale, bias, out,
                           M, N, K, R, nullptr, stream);
}

extern "C" int svdq_query_plan(int64_t M, int64_t N, int64_t K, int64_t R,
                               const svdq_options_t* options, int32_t sm_count,
                               svdq_plan_t* plan) {
  if (plan == nullptr) return SVDQ_ERR_INVALID_ARG;
  int rc = validate_options(options);
  if (rc != SVDQ_OK) return rc;
  if ((rc = validate_shape(M, N, K, R)) != SVDQ_OK) return rc;
  int smem = kGb300SmemOptin;
  if (sm_count <= 0) {
    int dev = 0;
    DeviceInfo* d = nullptr;
    if ((rc = probe_device(&dev, &d)) != SVDQ_OK) return rc;
    sm_count = d->sm_count;
    smem = d->smem_optin;
  }
  Plan pl;
  if ((rc = make_plan(M, N, K, R, options, sm_count, smem, 0, &pl,
                      options != nullptr && options->k_splits != 0)) != SVDQ_OK)
    return rc;
  std::memset(plan, 0, sizeof *plan);
  plan->tile_m = kBM * pl.cta_group;
  plan->tile_n = pl.tile_n;
  plan->tile_k = kBK;
  plan->cta_group = pl.cta_group;
  plan->num_ab_stage = pl.stages;
  plan->num_acc_stage = pl.acc_stages;
  plan->stage_bytes = pl.stage_bytes;
  plan->lora_block_bytes = pl.lora_block_bytes;
  plan->lora_blocks = pl.lora_blocks;
  plan->k_blocks = pl.k_blocks;
  plan->smem_bytes = pl.smem_bytes;
  plan->tmem_cols = kTmemCols;
  plan->tmem_cols_used = pl.tmem_cols_used;
  plan->threads = kThreads;
  plan->num_tiles = pl.num_tiles;
  plan->grid = pl.grid;
  plan->sm_count = sm_count;
  plan->kblocks_per_stage = pl.kbi;
  plan->k_splits = pl.splits;
  plan->num_units = pl.num_units;
  plan->workspace_bytes = ws_bytes(pl);
  return SVDQ_OK;
}

extern "C" int64_t svdq_lora_stage_bytes(int64_t tile_m, int64_t tile_n, int64_t R,
                                         int64_t elem_bytes, int64_t cta_group, int64_t* la_bytes,
                                         int64_t* lu_bytes) {
  if (tile_m <= 0 || tile_n <= 0 || R < 0 || elem_bytes <= 0 || cta_group <= 0 ||
      tile_m % cta_group || tile_n % cta_group)
    return SVDQ_ERR_INVALID_ARG;
  const int64_t la = tile_m * R * elem_bytes / cta_group;  // A side split along M
  const int64_t lu = tile_n * R * elem_bytes / cta_group;  // B side split along N
  if (la_bytes) *la_bytes = la;
  if (lu_bytes) *lu_bytes = lu;
  return la + lu;
}

extern "C" int svdq_read_device_status(int32_t* code, int32_t* site, int32_t* block, int clear) {
  int dev = 0;
  DeviceInfo* d = nullptr;
  int rc = probe_device(&dev, &d);
  if (rc != SVDQ_OK) return rc;
  int st[4] = {0, 0, 0, 0};
  if (cudaMemcpy(st, d->status, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return SVDQ_ERR_CUDA;
  }
  if (code) *code = st[0];
  if (site) *site = st[1];
  if (block) *block = st[2];
  if (clear) {
    const int zero[4] = {0, 0, 0, 0};
    if (cudaMemcpy(d->status, zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      return SVDQ_ERR_CUDA;
    }
    // a timed-out split launch may have left flags raised in the library's
    // scratch: start it from zero again
    void* scratch = nullptr;
    {
      std::lock_guard<std::mutex> lock(g_mutex);
      scratch = d->noalloc_scratch;
    }
    if (st[0] == SVDQ_ERR_TIMEOUT && scratch != nullptr &&
        (cudaMemset(scratch, 0, SVDQ_NOALLOC_SCRATCH_BYTES) != cudaSuccess ||
         cudaDeviceSynchronize() != cudaSuccess)) {
      cudaGetLastError();
      return SVDQ_ERR_CUDA;
    }
  }
  return SVDQ_OK;
}

extern "C" const char* svdq_status_string(int status) {
  switch (status) {
    case SVDQ_OK: return "SVDQ_OK";
    case SVDQ_ERR_INVALID_ARG: return "SVDQ_ERR_INVALID_ARG";
    case SVDQ_ERR_UNSUPPORTED_SHAPE: return "SVDQ_ERR_UNSUPPORTED_SHAPE";
    case SVDQ_ERR_MISALIGNED: return "SVDQ_ERR_MISALIGNED";
    case SVDQ_ERR_UNSUPPORTED_DEVICE: return "SVDQ_ERR_UNSUPPORTED_DEVICE";
    case SVDQ_ERR_LAUNCH: return "SVDQ_ERR_LAUNCH";
    case SVDQ_ERR_CUDA: return "SVDQ_ERR_CUDA";
    case SVDQ_ERR_TIMEOUT: return "SVDQ_ERR_TIMEOUT";
    case SVDQ_ERR_BAD_OPTION: return "SVDQ_ERR_BAD_OPTION";
    case SVDQ_ERR_WORKSPACE: return "SVDQ_ERR_WORKSPACE";
    case SVDQ_ERR_SCRATCH_LIMIT: return "SVDQ_ERR_SCRATCH_LIMIT";
    case SVDQ_ERR_WCSCALE_ZERO: return "SVDQ_ERR_WCSCALE_ZERO";
    case SVDQ_ERR_LU_OVERFLOW: return "SVDQ_ERR_LU_OVERFLOW";
    default: return "SVDQ_ERR_UNKNOWN";
  }
}

extern "C" int svdq_version(void) { return SVDQ_ABI_VERSION; }

extern "C" int svdq_w4a4_gemm_split_noalloc(const void* act, const void* wgt, const void* ascales,
                                            const void* wscales, const float* lora_act_in,
                                            const void* lora_up, const void* wcscale,
                                            const void* bias, void* out, int64_t M, int64_t N,
                                            int64_t K, int64_t R, const svdq_options_t* options,
                                            int32_t weights_prepacked, void* stream) {
  if (weights_prepacked != 0 && weights_prepacked != 1) return SVDQ_ERR_INVALID_ARG;
  // the plan's scratch need, computed exactly as the launch will plan
  const int64_t need = svdq_workspace_size(M, N, K, R, options, 0);
  if (need < 0) return static_cast<int>(need);
  if (need > SVDQ_NOALLOC_SCRATCH_BYTES) return SVDQ_ERR_SCRATCH_LIMIT;
  int dev = 0;
  DeviceInfo* d = nullptr;
  int rc = probe_device(&dev, &d);
  if (rc != SVDQ_OK) return rc;
  {
    // once per device, with that device current: the array's device address
    // (in host code the symbol is only a host-side stand-in)
    std::lock_guard<std::mutex> lock(g_mutex);
    if (d->noalloc_scratch == nullptr) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return SVDQ_ERR_CUDA;
      }
      d->noalloc_scratch = ptr;
    }
  }
  return run_gemm(act, wgt, ascales, wscales, lora_act_in, lora_up, wcscale, bias, out, M, N, K,
                  R, options, stream, weights_prepacked == 1, d->noalloc_scratch,
                  SVDQ_NOALLOC_SCRATCH_BYTES);
}

extern "C" int svdq_quantize_act(const void* x, const void* lora_down, int64_t M, int64_t K,
                                 int64_t R, int32_t io_dtype, int32_t scales_packed,
                                 int32_t lora_act_16bit, void* act, void* ascales,
                                 void* lora_act_in, void* stream) {
  using namespace svdq;
  int rc = validate_quant(x, lora_down, M, K, R, io_dtype, scales_packed, lora_act_16bit, act,
                          ascales, lora_act_in);
  if (rc != SVDQ_OK) return rc;
  if (M == 0) return SVDQ_OK;
  int dev = 0;
  DeviceInfo* dinfo = nullptr;
  if ((rc = probe_device(&dev, &dinfo)) != SVDQ_OK) return rc;
  QuantPlan qp;
  if ((rc = plan_quant(M, K, R, dinfo->sm_count, dinfo->smem_optin, &qp)) != SVDQ_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return io_dtype == SVDQ_IO_FP16
             ? launch_quant<true>(qp, dinfo, x, lora_down, M, K, R, scales_packed,
                                  lora_act_16bit, act, ascales, lora_act_in, s)
             : launch_quant<false>(qp, dinfo, x, lora_down, M, K, R, scales_packed,
                                   lora_act_16bit, act, ascales, lora_act_in, s);
}

extern "C" int svdq_quantize_query(int64_t M, int64_t K, int64_t R, int32_t sm_count,
                                   int32_t* splits, int32_t* grid, int32_t* stages,
                                   int32_t* smem_bytes) {
  using namespace svdq;
  if (M < 0 || K <= 0 || R < 0) return SVDQ_ERR_INVALID_ARG;
  if (M % 16 || K % 64 || M > SVDQ_MAX_MN || K > SVDQ_MAX_K || R > SVDQ_MAX_RANK)
    return SVDQ_ERR_UNSUPPORTED_SHAPE;
  int sms = sm_count, optin = kGb300SmemOptin;
  if (sms <= 0) {
    int dev = 0;
    DeviceInfo* dinfo = nullptr;
    const int rc = probe_device(&dev, &dinfo);
    if (rc != SVDQ_OK) return rc;
    sms = dinfo->sm_count;
    optin = dinfo->smem_optin;
  }
  QuantPlan qp;
  const int rc = plan_quant(M, K, R, sms, optin, &qp);
  if (rc != SVDQ_OK) return rc;
  if (splits) *splits = qp.splits;
  if (grid) *grid = qp.tiles * qp.splits;
  if (stages) *stages = qp.stages;
  if (smem_bytes) *smem_bytes = qp.smem;
  return SVDQ_OK;
}

extern "C" int64_t svdq_linear_workspace_size(int64_t M, int64_t K, int64_t R) {
  using namespace svdq;
  if (M < 0 || K <= 0 || R < 0) return SVDQ_ERR_INVALID_ARG;
  if (M % 16 || K % 64 || M > SVDQ_MAX_MN || K > SVDQ_MAX_K || R > SVDQ_MAX_RANK)
    return SVDQ_ERR_UNSUPPORTED_SHAPE;
  auto pad = [](int64_t b) { return (b + 255) / 256 * 256; };
  const int64_t la_bytes = R == 0 ? 0 : M * R * (R % 8 == 0 ? 2 : 4);
  return pad(M * K / 2) + pad(M * K / 16) + pad(la_bytes);
}

extern "C" int svdq_w4a4_linear(const void* x, const void* lora_down, const void* wgt,
                                const void* wscales_packed, const void* lora_up_packed,
                                const void* wcscale, const void* bias, void* out, int64_t M,
                                int64_t N, int64_t K, int64_t R, const svdq_options_t* options,
                                void* workspace, int64_t workspace_bytes, void* stream) {
  using namespace svdq;
  const int64_t need = svdq_linear_workspace_size(M, K, R);
  if (need < 0) return static_cast<int>(need);
  if (N < 0) return SVDQ_ERR_INVALID_ARG;
  if (N % 16 || N > SVDQ_MAX_MN) return SVDQ_ERR_UNSUPPORTED_SHAPE;
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)))
    return SVDQ_ERR_WORKSPACE;
  svdq_options_t o{};
  if (options != nullptr) o = *options;
  const int32_t la16 = (R > 0 && R % 8 == 0) ? 1 : 0;
  o.act_scales_packed = 1;
  o.lora_act_16bit = la16;
  // act [M][K/2], scale words [K/64][M], lora_act_in [M][R], each 256-byte aligned
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int64_t off_sc = (M * K / 2 + 255) / 256 * 256;
  const int64_t off_la = off_sc + (M * K / 16 + 255) / 256 * 256;
  void* act = ws;
  void* asc = ws != nullptr ? ws + off_sc : nullptr;
  void* la = (ws != nullptr && R > 0) ? ws + off_la : nullptr;
  int rc = svdq_quantize_act(x, lora_down, M, K, R, o.io_dtype, 1, la16, act, asc, la, stream);
  if (rc != SVDQ_OK) return rc;
  return svdq_w4a4_gemm_prepacked(act, wgt, asc, wscales_packed, static_cast<const float*>(la),
                                  lora_up_packed, wcscale, bias, out, M, N, K, R, &o, stream);
}
