"""Plain CPU oracle of the routed mixture-of-experts layer forward.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this package.  The library's own
path never calls it, and the two share no code.  Both sides read the same
seeded inputs from the `synth` module.

The oracle is slow and obviously correct.  It is plain numpy.  Layer
arithmetic (dequantisation, SwiGLU, combine) runs in fp64.  Where floating
point decides an integer, the oracle decides it in fp32, in the order this
library defines:
  * the router logits that choose the top-k ids;
  * the activation codes of the prefill mirror.

Modules:
  formats  - E2M1 / E4M3 / E8M0 / bf16 decoding, weight dequantisation,
             activation quantisation (prefill mirror)
  route    - router logits in the library's fixed fp32 order, softmax, top-k
  permute  - stable expert-sorted permutation
  ffn      - grouped SwiGLU expert FFN, weighted combine, whole layer
  lru      - global LRU slot map over (layer, expert) keys

Parity status: every function is pinned by the `-m "not gpu"` tests in
tests/test_oracle_*.py against closed forms, library routines, brute force
or hand-derived golden values.  The softmax weights are pinned against
scipy.special.softmax and the two-expert sigmoid; the SiLU against
scipy.special.expit, sigmoid(ln 3) = 3/4 and silu(g) - silu(-g) = g.
The prefill mirror (ffn.swiglu with act_quant, ffn._mirror and the
formats.quant_act_* / dequant_act_* pairs it uses) is pinned by hand-derived
examples in tests/golden/mirror_examples.json: one expert with a diagonal gate
and permutation up/down matrices in NVFP4 and FP8, two scale blocks each,
checked step by step; planted mistakes (h or x not quantised, g quantised
instead of h, a transposed operand, a divided or interleaved scale) each
change the result (tests/test_oracle_mirror.py).
"""
from . import formats, route, permute, ffn, lru  # noqa: F401
