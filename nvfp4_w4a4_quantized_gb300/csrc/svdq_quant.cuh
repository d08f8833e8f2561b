// svdq_quant.cuh -- the activation-side producer of the W4A4 operator's inputs
// ("SVDQuant W4A4 on Blackwell" §1: the operator is the compute-bound half of
// SVDQuant; §2: act, ascales and lora_act_in are its activation inputs, with
// LA the LoRA-down activation of §3.3).  One pass over 16-bit activations x
// [M, K] writes
//   act[m, k/2]      E2M1 codes, low nibble = even k          (NVFP4 values)
//   ascales[k/16, m] E4M3 group scales (or the packed words [k/64, m])
//   lora_act_in[m,r] = sum_k x[m, k] * lora_down[r, k]        (fp32)
// with, per group of 16 consecutive k in a row,
//   s = E4M3_RNE_satfinite(amax / 6),   code = E2M1_RNE_satfinite(x / s),
// amax the group's largest |x|, and every code 0 where s == 0.  A value that
// rounds to zero is stored as +0 (code 0) whatever its sign.
//
// Kernel layout, one CTA per 128-row tile and K range (a cluster of `splits`
// CTAs shares a row tile along K and adds its LoRA-down partials through
// distributed shared memory, in rank order):
//   warp 0      TMA producer (one thread): per 64-wide K chunk the x box
//               [128 rows x 128 bytes] and the lora_down box [R16 rows x 128
//               bytes], both with the 128-byte swizzle, into a ring of stages.
//   warp 1      tensor-memory allocation; one thread issues the LoRA-down MMAs
//               (tcgen05.mma kind::f16, M = 128, N = R16, four K = 16 steps per
//               chunk) into a fp32 accumulator in tensor memory.
//   warps 2..17 quantisers, one row per lane: warp 2 + 4h + q takes rows
//               32q .. 32q + 31 of chunks h, h + 4, h + 8, ... (four chunks in
//               work at once, so that the dependent arithmetic of one chunk
//               overlaps the others'); per chunk a lane writes its row's 32
//               code bytes and 4 scale bytes.  Warps 2..5 then read the
//               accumulator back (lane quadrant = warp % 4).
// Every wait is bounded (globaltimer) and reports SVDQ_ERR_TIMEOUT through the
// device status word instead of hanging.
#pragma once

#include "svdq_kernel.cuh"

namespace svdq {

constexpr int kQThreads = 576;   // 18 warps
constexpr int kQRows = 128;      // rows per tile (the MMA's M)
constexpr int kQChunk = 64;      // K elements per ring stage: 128 bytes of x per row
constexpr int kQXBytes = kQRows * 128;
constexpr int kQMaxStages = 12;
constexpr int kQMaxSplits = 8;

enum QuantWaitSite : int {
  kSiteQuantEmpty = 11,
  kSiteQuantFull = 12,
  kSiteQuantMma = 13,
  kSiteQuantAcc = 14,
};

struct QParams {
  uint8_t* act;       // [M, K/2]
  uint8_t* ascales;   // [K/16, M] bytes, or uint32 [K/64, M] words when packed
  void* la;           // [M, R] fp32, or 16-bit (la16) in x's type; null when R == 0
  int la16;           // lora_act_in as 16-bit values (RNE from the fp32 sum)
  int M, K, R, r16;   // r16 = R rounded up to 16 (0 without LoRA)
  int chunks;         // K / 64
  int splits;         // CTAs per row tile (the cluster size), 1..8
  int stages;
  int packed;
  int tmem_cols;
  int* status;
  unsigned long long timeout_ns;
};

// Shared-memory layout (offsets from the 1024-aligned base).
__host__ __device__ constexpr int quant_stage_bytes(int r16) { return kQXBytes + 128 * r16; }
__host__ __device__ constexpr int quant_part_pitch(int r16) { return r16 + 4; }  // floats
// The cluster's LoRA-down partials [128][R16 + 4] fp32 reuse the ring's stages
// once every chunk has been consumed.
__host__ __device__ constexpr int quant_part_bytes(int r16) {
  return kQRows * quant_part_pitch(r16) * 4;
}
__host__ __device__ constexpr int quant_smem_bytes(int r16, int stages) {
  return 1024 + stages * quant_stage_bytes(r16) + 8 * (2 * kQMaxStages + 1) + 16 +
         128 * 8;  // barriers, TMEM slot, flag, scale table
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Columns col .. col + n - 1 (n = 4 or 1) of lora_act_in row `row`: fp32, or
// 16-bit (RNE) with la16.  n = 4 needs R % 4 == 0 (8- or 16-byte aligned rows).
template <bool F16>
__device__ __forceinline__ void store_la(const QParams& p, int row, int col, float4 v, int n) {
  const size_t at = static_cast<size_t>(row) * p.R + col;
  if (p.la16) {
    uint16_t* dst = static_cast<uint16_t*>(p.la) + at;
    if (n == 4) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(H16<F16>::pack(v.x, v.y), H16<F16>::pack(v.z, v.w));
    } else {
      *dst = static_cast<uint16_t>(H16<F16>::pack(v.x, 0.0f) & 0xFFFFu);
    }
  } else {
    float* dst = static_cast<float*>(p.la) + at;
    if (n == 4)
      *reinterpret_cast<float4*>(dst) = v;
    else
      *dst = v.x;
  }
}

// Largest |x| of 16 values given as eight 16-bit pairs (finite values).
template <bool F16>
__device__ __forceinline__ float group_amax(const uint32_t* w) {
  const uint32_t m01 = ptx::maxabs16x2<F16>(w[0], w[1]), m23 = ptx::maxabs16x2<F16>(w[2], w[3]);
  const uint32_t m45 = ptx::maxabs16x2<F16>(w[4], w[5]), m67 = ptx::maxabs16x2<F16>(w[6], w[7]);
  const uint32_t m = ptx::maxabs16x2<F16>(ptx::maxabs16x2<F16>(m01, m23),
                                          ptx::maxabs16x2<F16>(m45, m67));
  return H16<F16>::lo(ptx::maxabs16x2<F16>(m, m >> 16) & 0x7FFFu);
}

// Correctly rounded a / b from rcp = RN(1/b): q0 = RN(a rcp) is within an ulp
// of a / b; the residual a - q0 b is exact in one fma, and one Newton-Raphson
// step on it (Markstein's correction) returns RN(a / b).
__device__ __forceinline__ float div_markstein(float a, float b, float rcp) {
  const float q0 = __fmul_rn(a, rcp);
  return __fmaf_rn(__fmaf_rn(-q0, b, a), rcp, q0);
}

// One group of 16: returns the scale byte and writes the 8 code bytes (two
// words; byte i = elements 2i (low nibble) and 2i + 1).  `tab` holds, per
// E4M3 byte with value s, 1/s as an unevaluated sum hi + lo of two fp32
// (hi = RN(1/s), lo = RN(1/s - hi)); both 0 for s = 0.
template <bool F16>
__device__ __forceinline__ uint32_t quant_group(const uint32_t* w, const float2* tab,
                                                uint32_t* codes) {
  constexpr float kRcp6 = 1.0f / 6.0f;  // RN(1/6)
  const uint32_t sb = ptx::cvt_e4m3(div_markstein(group_amax<F16>(w), 6.0f, kRcp6));
  const float2 inv = tab[sb];
  // The code is that of the exact quotient x / s.  q = RN(x hi + RN(x lo))
  // is x / s to about 2^-47 (relative): on an E2M1 tie exactly when x / s is
  // (ties are representable), and otherwise on the same side of every
  // rounding boundary (a 16-bit x over an E4M3 s is at least 2^-11, relative,
  // away from one).  s == 0 gives quotients 0 and codes 0.  Pairs of elements
  // go through the packed fp32x2 pipe.
  const uint64_t hi2 = ptx::f32x2(inv.x, inv.x);
  const uint64_t lo2 = ptx::f32x2(inv.y, inv.y);
#pragma unroll
  for (int hw = 0; hw < 2; ++hw) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t x2 = w[4 * hw + i];
      const uint64_t xx = ptx::f32x2(H16<F16>::lo(x2), H16<F16>::hi(x2));
      const uint64_t q = ptx::fma_f32x2(xx, hi2, ptx::mul_f32x2(xx, lo2));
      ptx::f32x2_split(q, v[2 * i], v[2 * i + 1]);
    }
    const uint32_t word = ptx::cvt_e2m1x8(v);
    // a code whose magnitude is zero is stored as +0
    const uint32_t mag = word & 0x77777777u;
    const uint32_t nonzero = (mag + 0x77777777u) & 0x88888888u;
    codes[hw] = word & (nonzero | 0x77777777u);
  }
  return sb;
}

template <bool F16>
__global__ void __launch_bounds__(kQThreads, 1)
    svdq_quant_kernel(const __grid_constant__ CUtensorMap tm_x,
                      const __grid_constant__ CUtensorMap tm_ld, const QParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = static_cast<int>(threadIdx.x) / 32;
  const int lane = static_cast<int>(threadIdx.x) % 32;
  const int S = p.stages;
  const int split = p.splits > 1 ? static_cast<int>(ptx::cluster_ctarank()) : 0;
  const int tile = static_cast<int>(blockIdx.x) / p.splits;
  const int c_begin = split * p.chunks / p.splits;
  const int n = (split + 1) * p.chunks / p.splits - c_begin;
  const bool lora = p.r16 > 0;
  const int stage_bytes = quant_stage_bytes(p.r16);
  const uint32_t part_base = sbase;  // over the stages, after the last chunk
  uint8_t* bar_area = smem + S * stage_bytes;
  const uint32_t bar0 = ptx::smem_u32(bar_area);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kQMaxStages + s); };
  const uint32_t acc_full = bar0 + 8u * (2 * kQMaxStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 8 * (2 * kQMaxStages + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const Ctl ctl{abort_flag, p.status, p.timeout_ns};
  // E4M3 byte -> 1/value as hi + lo; 0x7F (NaN) is never produced
  float2* scale_tab = reinterpret_cast<float2*>(bar_area + 8 * (2 * kQMaxStages + 1) + 16);
  // built by warps 2..5 while thread 0 starts the ring
  if (threadIdx.x >= 64 && threadIdx.x < 64 + 128) {
    const uint32_t b = threadIdx.x - 64;
    const float v = b < 0x7F ? ptx::e4m3_value(b) : 0.0f;
    const float hi = v > 0.0f ? __frcp_rn(v) : 0.0f;
    // 1 - v hi is exact in one fma (v has 4 significant bits); times hi it is
    // 1/v - hi to fp32 precision
    const float lo = __fmul_rn(__fmaf_rn(-v, hi, 1.0f), hi);
    scale_tab[b] = make_float2(hi, v > 0.0f ? lo : 0.0f);
  }

  // Thread 0 is the producer: it sets up the barriers and issues the ring's
  // first S loads (every stage starts empty) before the CTA-wide barrier, so
  // the first chunks are in flight while the rest of the set-up runs.
  const uint32_t load_bytes = static_cast<uint32_t>(kQXBytes + (lora ? 128 * p.r16 : 0));
  auto issue = [&](int i) {
    const int stage = i % S;
    const uint32_t st = sbase + stage * stage_bytes;
    const int kx = (c_begin + i) * kQChunk;
    ptx::mbar_arrive_expect_tx(full(stage), load_bytes);
    ptx::tma_load_2d(st, &tm_x, full(stage), kx, tile * kQRows);
    if (lora) ptx::tma_load_2d(st + kQXBytes, &tm_ld, full(stage), kx, 0);
  };
  const int pre = n < S ? n : S;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(full(s), 1);                  // the producer's byte count
      ptx::mbar_init(empty(s), 16 + (lora ? 1 : 0));  // every quantiser warp + the MMA commit
    }
    ptx::mbar_init(acc_full, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tm_x);
    if (lora) ptx::prefetch_tmap(&tm_ld);
    // x is read only once the previous kernel of the stream has completed
    ptx::griddep_wait();
    for (int i = 0; i < pre; ++i) issue(i);
  }
  if (warp == 1 && lora) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), static_cast<uint32_t>(p.tmem_cols));
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  // Programmatic stream serialisation: nothing in global memory is touched
  // before the previous kernel of the stream has completed.
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = pre;
      for (int i = pre; i < n; ++i) {
        // the stage's previous chunk (i - S) has been released
        if (!wait_bar<false>(empty(i % S), static_cast<uint32_t>(((i / S) & 1) ^ 1),
                             kSiteQuantEmpty, ctl))
          break;
        issue(i);
        ++issued;
      }
      // every copy this thread started has landed before the CTA can exit
      for (int j = issued > S ? issued - S : 0; j < issued; ++j)
        drain_wait(full(j % S), static_cast<uint32_t>((j / S) & 1));
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ LoRA-down MMA
    if (lora && lane == 0) {
      const uint32_t idesc = F16 ? ptx::idesc_f16_f32(kQRows, static_cast<uint32_t>(p.r16))
                                 : ptx::idesc_bf16_f32(kQRows, static_cast<uint32_t>(p.r16));
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        if (!wait_bar<false>(full(stage), phase, kSiteQuantMma, ctl)) {
          ok = false;
          break;
        }
        ++issued;
        ptx::tc_fence_after();
        const uint32_t xs = sbase + stage * stage_bytes;
#pragma unroll
        for (int s = 0; s < 4; ++s)
          ptx::mma_bf16(tmem_base, ptx::desc_kmajor_sw128(xs + 32 * s),
                        ptx::desc_kmajor_sw128(xs + kQXBytes + 32 * s), idesc,
                        (i > 0 || s > 0) ? 1u : 0u);
        ptx::mma_commit(empty(stage));
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // the accumulator is complete (or, after an abort, every MMA issued
      // has finished with shared and tensor memory before the teardown)
      if (issued > 0) {
        ptx::mma_commit(acc_full);
        if (!ok) drain_wait(acc_full, 0u);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ quantisers
    const int q = warp & 3;
    // This warp quantises chunks h, h + 4, h + 8, ... (four chunks in work at
    // once).  It still waits on every chunk's full barrier in order and signs
    // every chunk's release, so it can never fall two phases behind on a
    // barrier it tracks by parity, whatever the ring depth.
    const int h = (warp - 2) >> 2;
    const int r = 32 * q + lane;    // row within the tile (= tensor-memory lane)
    const int grow = tile * kQRows + r;
    const bool live = grow < p.M;
    const int sw = r & 7;  // 128-byte swizzle: 16-byte piece j of row r sits at j ^ (r % 8)
    uint8_t* act_row = p.act + static_cast<size_t>(grow) * static_cast<size_t>(p.K / 2);
    bool ok = true;
    int stage = 0;
    uint32_t phase = 0;
    for (int i = 0; i < n; ++i) {
      if (!warp_wait_bar<false>(full(stage), phase, kSiteQuantFull, ctl)) {
        ok = false;
        break;
      }
      if ((i & 3) == h) {
        const uint8_t* xr = smem + stage * stage_bytes + r * 128;
        uint32_t codes[8], sb[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint4 a = lds128(xr + (((2 * g) ^ sw) << 4));
          const uint4 b = lds128(xr + (((2 * g + 1) ^ sw) << 4));
          const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
          sb[g] = quant_group<F16>(w, scale_tab, codes + 2 * g);
        }
        // the stage goes back to the producer once every lane has used its
        // loaded words (a load is complete once its value has been consumed)
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty(stage));
        if (live) {
          const int c = c_begin + i;
          uint4* dst = reinterpret_cast<uint4*>(act_row + 32 * c);
          dst[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
          dst[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
          if (p.packed) {
            reinterpret_cast<uint32_t*>(p.ascales)[static_cast<size_t>(c) * p.M + grow] =
                sb[0] | (sb[1] << 8) | (sb[2] << 16) | (sb[3] << 24);
          } else {
#pragma unroll
            for (int g = 0; g < 4; ++g)
              p.ascales[static_cast<size_t>(4 * c + g) * p.M + grow] = static_cast<uint8_t>(sb[g]);
          }
        }
      } else if (lane == 0) {
        ptx::mbar_arrive(empty(stage));
      }
      if (++stage == S) {
        stage = 0;
        phase ^= 1u;
      }
    }
    // every quantiser has finished with the stages (the partials reuse them)
    asm volatile("bar.sync 1, %0;" ::"n"(16 * 32) : "memory");
    if (lora && h == 0) {
      // ---------------------------------------------------------- LoRA-down readback
      const bool got = ok && warp_wait_bar<false>(acc_full, 0u, kSiteQuantAcc, ctl);
      if (got) {
        ptx::tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
        for (int c0 = 0; c0 < p.r16; c0 += 16) {
          uint32_t v[16];
          ptx::tmem_ld_32x32b_x8(taddr + c0, v);
          ptx::tmem_ld_32x32b_x8(taddr + c0 + 8, v + 8);
          ptx::tmem_wait_ld();
          if (p.splits == 1) {
            if (live) {
              if ((p.R & 3) == 0 && c0 + 16 <= p.R) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  store_la<F16>(p, grow, c0 + 4 * j,
                                make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                            __uint_as_float(v[4 * j + 2]),
                                            __uint_as_float(v[4 * j + 3])),
                                4);
              } else {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  if (c0 + j < p.R)
                    store_la<F16>(p, grow, c0 + j,
                                  make_float4(__uint_as_float(v[j]), 0.0f, 0.0f, 0.0f), 1);
              }
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(
                smem + 4 * (r * quant_part_pitch(p.r16) + c0));
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                   __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
          }
        }
      }
    }
  }

  // Every role is done with tensor memory and, for a cluster, the partials
  // are in place.  The cluster barriers are taken by every thread of every CTA.
  __syncwarp();
  ptx::tc_fence_before();
  if (p.splits > 1)
    ptx::cluster_sync();
  else
    __syncthreads();
  ptx::tc_fence_after();
  if (lora && p.splits > 1) {
    // rank `split` adds rows [split * 128 / splits, ...) over the cluster, rank order
    const int rows = kQRows / p.splits;
    const int row0 = split * rows;
    const int pitch = quant_part_pitch(p.r16);
    // four consecutive ranks per thread when rows stay aligned (R % 4 == 0), else one
    const int vec = (p.R & 3) == 0 ? 4 : 1;
    const int per_row = p.R / vec;
    for (int e = static_cast<int>(threadIdx.x); e < rows * per_row; e += kQThreads) {
      const int rr = row0 + e / per_row;
      const int col = vec * (e % per_row);
      const uint32_t a = part_base + 4u * static_cast<uint32_t>(rr * pitch + col);
      // all loads first (one distributed-shared-memory latency), then the
      // sum in rank order
      float4 part[kQMaxSplits];
#pragma unroll
      for (int s = 0; s < kQMaxSplits; ++s) {
        part[s] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (s < p.splits) {
          const uint32_t ra = ptx::mapa(a, static_cast<uint32_t>(s));
          if (vec == 4)
            part[s] = ld_cluster_f32x4(ra);
          else
            part[s].x = ld_cluster_f32(ra);
        }
      }
      float4 acc = part[0];
#pragma unroll
      for (int s = 1; s < kQMaxSplits; ++s) {
        if (s < p.splits) {
          acc.x += part[s].x;
          acc.y += part[s].y;
          acc.z += part[s].z;
          acc.w += part[s].w;
        }
      }
      const int grow = tile * kQRows + rr;
      if (grow < p.M) store_la<F16>(p, grow, col, acc, vec);
    }
    // no CTA leaves while a peer may still read its partials
    __syncwarp();
    ptx::cluster_sync();
  }
  if (warp == 1 && lora) ptx::tmem_dealloc(tmem_base, static_cast<uint32_t>(p.tmem_cols));
}

}  // namespace svdq
