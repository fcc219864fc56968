// Counter-based uniforms and the Gumbel perturbation used to draw the next
// token ("Kernels, Fusion & CUDA Graphs", "Fix 1: kernel fusion", the
// "Sampling" row: softmax, top-k / top-p and the draw in the kernel that has
// the logits).
//
// The generator is Philox4x32 with 10 rounds (Salmon, Moraes, Dror and Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC 2011), written from its
// published round function: the counter (c0, c1, c2, c3) becomes
// (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)) and the
// key advances by (W0, W1) after every round but the last. The draw for
// token `id` of batch row `row` at step `step` uses counter
// (id, row, step mod 2^32, step div 2^32) and key (seed mod 2^32, seed div
// 2^32); its first word x gives u = (floor(x / 512) + 1/2) * 2^-23 (24
// significant bits: exact in fp32) and the Gumbel variate -log(-log(u)).
#pragma once
#include <stdint.h>

#include "internal.h"

namespace mbt {

__device__ __forceinline__ uint32_t philox_first_word(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                      uint32_t k0, uint32_t k1) {
  constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u, W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += W0; k1 += W1; }
    const uint32_t hi0 = __umulhi(M0, c0), lo0 = M0 * c0;
    const uint32_t hi1 = __umulhi(M1, c2), lo1 = M1 * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
  }
  return c0;
}

// Temperature-scaled logit plus the token's Gumbel variate: the arg-max of
// this over a set of tokens is a draw from softmax(logit / T) over that set.
__device__ __forceinline__ float gumbel_score(float logit, int id, int row, const GumbelArgs& g) {
  const uint32_t x = philox_first_word((uint32_t)id, (uint32_t)(row + g.row0), g.step_lo, g.step_hi, g.seed_lo,
                                       g.seed_hi);
  const float u = ((float)(x >> 9) + 0.5f) * 1.1920928955078125e-7f;   // 2^-23
  return logit * g.inv_t - logf(-logf(u));
}

}  // namespace mbt
