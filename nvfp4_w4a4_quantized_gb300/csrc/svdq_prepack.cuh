// svdq_prepack.cuh -- weight-side prepack ("SVDQuant W4A4 on Blackwell" §3.1
// block scales per 64-wide MMA step, §6.3 LoRA sharing the main accumulator).
//
// Two independent element-wise passes in one grid-stride launch, both bound
// by HBM bandwidth and run once per weight load:
//   1. packed scale words: word (s, n) of uint32 [K/64][N] carries the group
//      scales wscales[4s .. 4s+3][n] in bytes 0..3.  A thread reads 4 bytes of
//      each of the 4 group rows for columns n .. n+3 (coalesced across
//      threads), transposes them in registers and writes 16 bytes.
//   2. LU' = round16(fp32(LU) * rcp(wcscale)): the correctly rounded fp32
//      reciprocal and product the fused kernel would otherwise compute per
//      call, rounded (RNE) into the 16-bit I/O type.  A zero wcscale (LU' set
//      to 0: that column's LoRA term is lost) or an LU' beyond the 16-bit
//      range is recorded in the device status word, as in the fused kernel.
#pragma once

#include "svdq_kernel.cuh"

namespace svdq {

template <bool F16>
__global__ void __launch_bounds__(256)
    svdq_prepack_kernel(const uint8_t* __restrict__ wscales, const uint16_t* __restrict__ lu,
                        const uint16_t* __restrict__ wc, uint32_t* __restrict__ wpk,
                        uint16_t* __restrict__ lup, int N, int K, int R, int* status) {
  using H = H16<F16>;
  const long long quads = static_cast<long long>(N / 4);
  const long long n_words = static_cast<long long>(K / 64) * quads;
  const long long n_lu = static_cast<long long>(N) * R;
  const long long total = n_words + n_lu;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    if (i < n_words) {
      const int s = static_cast<int>(i / quads);
      const int c = 4 * static_cast<int>(i - s * quads);
      const uint8_t* src = wscales + static_cast<size_t>(4 * s) * N + c;
      const uint32_t g0 = __ldg(reinterpret_cast<const uint32_t*>(src));
      const uint32_t g1 = __ldg(reinterpret_cast<const uint32_t*>(src + N));
      const uint32_t g2 = __ldg(reinterpret_cast<const uint32_t*>(src + 2 * N));
      const uint32_t g3 = __ldg(reinterpret_cast<const uint32_t*>(src + 3 * N));
      // byte j of group row g (column c + j) -> byte g of word j
      const uint32_t t0 = __byte_perm(g0, g1, 0x5140);
      const uint32_t t1 = __byte_perm(g0, g1, 0x7362);
      const uint32_t t2 = __byte_perm(g2, g3, 0x5140);
      const uint32_t t3 = __byte_perm(g2, g3, 0x7362);
      uint4 w;
      w.x = __byte_perm(t0, t2, 0x5410);
      w.y = __byte_perm(t0, t2, 0x7632);
      w.z = __byte_perm(t1, t3, 0x5410);
      w.w = __byte_perm(t1, t3, 0x7632);
      *reinterpret_cast<uint4*>(wpk + static_cast<size_t>(s) * N + c) = w;
    } else {
      const long long e = i - n_words;
      const int n = static_cast<int>(e / R);
      float inv = 1.f;
      if (wc != nullptr) {
        const float w = H::one(__ldg(wc + n));
        inv = (w != 0.f) ? __frcp_rn(w) : 0.f;
        if (w == 0.f) report_lora_operand(status, kStatusWcscaleZero, n);
      }
      const float v = __fmul_rn(H::one(__ldg(lu + e)), inv);
      const uint32_t h = H::pack(v, 0.f);
      if (nonfinite16_bits<F16>(h & 0xFFFFu)) report_lora_operand(status, kStatusLuOverflow, n);
      lup[e] = static_cast<uint16_t>(h & 0xFFFFu);
    }
  }
}

}  // namespace svdq
