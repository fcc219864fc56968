"""Oracle: a plain, slow, fp64 CPU implementation of one decode step of a dense
Llama-style decoder with a paged KV cache.

TEST INFRASTRUCTURE ONLY. Only the test suite, the package's smoke check and the
benchmark's CPU-baseline leg may import this package. The product path (the CUDA
library and its Python binding) never imports it and shares no code with it.

Pinning status (what ties each function to something other than itself; the
pins live in tests/test_oracle_*.py):

* numerics.bf16_decode / e4m3_decode: bit patterns with values fixed by the
  formats' definitions (1.0, 448, the smallest subnormal, NaN codes).
* numerics.round_bf16 / round_e4m3: exhaustive round-trip over every code,
  midpoints between neighbours (ties to even), saturation at +-448.
* decode.rmsnorm: unit RMS output at gamma = 1, scale invariance.
* decode.rope: pair rotation by a hand-checked 2-D rotation, per-pair angle
  p * theta^(-2i/d) read back with atan2, norm preservation, relative-position
  invariance of q.k, identity at p = 0.
* decode.silu / swiglu: silu(0) = 0, silu(1) = 1/(1+e^-1), silu(x) -> x and
  silu(-x) -> 0 for large x.
* decode.paged_attention: brute-force softmax over a contiguous cache written
  as plain Python loops, shuffled block tables, S in {1, 15, 16, 17, 33},
  GQA groups 1, 2, 5, 8; S = 1 gives V_0; q = 0 gives the mean of V.
* decode.prefill: the same logits and cache as feeding the prompt to
  decode_step one token at a time (the definition), on tiny models, from
  position 0 and from a later start.
* decode.decode_step: a scalar pure-Python brute-force step on a tiny model;
  closed forms with zeroed projections (logits = W_lm . norm(E[tok]));
  shift invariance of the whole step under a common position offset; the
  per-token multiply-add count within 1 % of 2 x matmul params + attention,
  within 10 % of 2 x all params.

* sampling.philox4x32_10: the generator's published known-answer vectors
  (tests/golden/philox4x32_10_kat.json); sampling.uniforms: values strictly
  inside (0, 1) on the 2^-23 grid, moments and a chi-square test of
  uniformity; sampling.sample: Gumbel-max frequencies against softmax
  probabilities (chi-square), arg-max at top_k = 1, at a vanishing temperature
  and at a tiny top_p, draws inside the top-k set; sampling.keep_set: the
  top-p set is the minimal most-probable prefix.

No function is "parity unpinned".
"""
from . import numerics, decode, sampling  # noqa: F401
